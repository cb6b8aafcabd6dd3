// fused.cu -- a decode-size (T <= 32) MoE layer, or a stack of them with
// RMSNorm and the residual between layers, as ONE persistent kernel.
//
// The pages trace decode time to launches and to per-stage waits: router
// top-k and grouping, the shared expert and the MoE end each got their own
// launch and were then fused (Strata, "Qwen3.6-35B-A3B: pictures, several
// requests at once and speed", section "Speed"); a whole layer's experts go
// through one launch per stage (PolyStrata, "Models and backends", section
// "What was tuned").  Here the stages of every layer are phases of one
// cooperative kernel with one CTA per SM, separated by grid barriers:
//
//   x  every CTA stages the layer's activations in shared memory (in a
//      stack: bf16(rmsnorm(resid)), the norm's sums of squares coming from
//      the previous layer's per-CTA partial sums)
//   A  router rows (E+1: the last is the shared-expert gate) and the shared
//      expert's gate/up rows, spread over the CTAs -> logits, shared SwiGLU
//   -- barrier --
//   B  every CTA selects each token's top-K from the logits and buckets the
//      (token, k) pairs by expert (the same result everywhere); then its
//      contiguous share of the touched experts' gate/up row pairs -> h
//   -- barrier --
//   C  every CTA owns a block of output rows: the shared expert's and every
//      touched expert's down rows for that block against the SwiGLU vectors
//      of their slots, then the weighted combine (and, in a stack, the
//      residual update and its partial sums of squares)
//   -- barrier (stack only) --
//
// All weights reach shared memory through one ring of fixed-size slots fed
// by a producer thread with 1-D bulk copies (cp.async.bulk) completing on
// mbarriers.  The producer walks the chunks in the order the consumer warps
// use them: a layer's router rows and shared gate/up pairs need no routing,
// so they are requested as soon as slots free up -- during the previous
// layer's gate/up and down phases in a stack; the routed gate/up pairs and
// the down rows follow as soon as the CTA has routed the layer, and the
// SwiGLU vectors the down rows meet are copied into the same chunks right
// after the second barrier.  Each phase is one non-inlined routine, so its
// instructions are fetched once per layer whatever the call site.  Every
// wait is bounded; a wait that runs out latches STRATA_ETIMEOUT.

#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "route.cuh"

namespace strata {

static_assert(sizeof(FusedLaunch) <= 4096, "kernel parameters beyond 4 KB");

constexpr int kFxConsumers = 8;
constexpr int kFxThreads = 32 * (kFxConsumers + 1);
constexpr int kFxPairs = 8;          // gate/up row pairs per chunk
constexpr int kFxMaxItems = 16;      // down-phase items per chunk
constexpr int NW = kFxConsumers, NCT = kFxConsumers * 32;

// Synchronises the consumer warps only (named barrier 1).
struct ConsSync {
    __device__ void operator()() const {
        asm volatile("bar.sync 1, %0;" ::"r"(kFxConsumers * 32) : "memory");
    }
};

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long global_clock() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Generic-proxy global writes made visible to later bulk copies (the async
// proxy) of this or other CTAs.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Adds to an mbarrier phase's expected transaction bytes without arriving.
__device__ __forceinline__ void mbar_expect_tx_only(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// try_wait that lets the hardware park the thread for up to `ns`
// nanoseconds or until the phase completes.
__device__ __forceinline__ bool mbar_try_wait_park(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded mbarrier wait of ONE thread (parked between polls, so a waiting
// warp takes no issue slots and no shared-memory bandwidth from the warps
// at work or from the bulk copies landing); it also gives up early once
// another wait of the kernel has run out (so one lost arrival costs one
// time limit, not one per remaining wait).
__device__ __forceinline__ bool fx_wait(uint64_t* bar, uint32_t parity, const uint32_t* err) {
#pragma unroll 1
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait_park(bar, parity, 1000u)) return true;
        if ((i & 255u) == 255u && *reinterpret_cast<const volatile uint32_t*>(err) == 4u)
            return false;
    }
    return false;
}

// Grid barrier of the consumer warps of every CTA (all co-resident: the
// kernel is launched cooperatively).  CTA 0 adds 2^31 - (G - 1), every
// other CTA 1, so the top bit of the word flips exactly when the last CTA
// arrives and the low bits are back to 0 afterwards.
__device__ __noinline__ void fx_grid_sync(uint32_t* bar, uint32_t* err, int ct, uint32_t site,
                                          uint32_t item) {
    ConsSync{}();
    if (ct == 0) {
        __threadfence();
        const uint32_t add = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1u) : 1u;
        const uint32_t old = atomicAdd(bar, add);
        uint32_t n = 0;
        while (((ld_acquire_gpu(bar) ^ old) & 0x80000000u) == 0u) {
            if (++n >= kWaitLimit) {
                latch_timeout(err, site, 0, 0, item);
                break;
            }
            if ((n & 255u) == 0u && *reinterpret_cast<const volatile uint32_t*>(err) == 4u) break;
        }
        __threadfence();
    }
    ConsSync{}();
}

// ------------------------------------------------------------------ ring
// trace: NULL, or (profiling, one thread of CTA 0) the clock of every
// chunk's issue [k], arrival [64 + k] and release [128 + k], k < 64.
struct Ring {
    uint8_t* base;
    uint64_t* full;
    uint64_t* empty;
    uint32_t S, SB;
    uint32_t* err;
    unsigned long long* trace;
};
constexpr uint32_t kFxTraceChunks = 64;

// Consumer side: lane 0 waits for chunk k, the warp follows (__syncwarp
// orders the lanes' reads after lane 0's acquire of the bulk copies).
__device__ __forceinline__ const uint8_t* ring_wait(const Ring& R, uint32_t k, int lane) {
    const uint32_t slot = k % R.S, round = k / R.S;
    if (lane == 0 && !fx_wait(&R.full[slot], round & 1u, R.err))
        latch_timeout(R.err, 23, slot, round, k);
    __syncwarp();
    if (R.trace != nullptr && k < kFxTraceChunks) R.trace[kFxTraceChunks + k] = global_clock();
    return R.base + size_t(slot) * R.SB;
}

__device__ __forceinline__ void ring_release(const Ring& R, uint32_t k, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[k % R.S]);
    if (R.trace != nullptr && k < kFxTraceChunks) R.trace[2 * kFxTraceChunks + k] = global_clock();
}

// Producer side: waits until slot k % S is free.
__device__ __forceinline__ uint8_t* ring_acquire(const Ring& R, uint32_t k) {
    const uint32_t slot = k % R.S, round = k / R.S;
    if (round > 0 && !fx_wait(&R.empty[slot], (round - 1) & 1u, R.err))
        latch_timeout(R.err, 21, slot, round, k);
    if (R.trace != nullptr && k < kFxTraceChunks) R.trace[k] = global_clock();
    return R.base + size_t(slot) * R.SB;
}

// ----------------------------------------------------------- activations
// The layer's activations in shared memory, bf16, in an order that makes a
// lane's read of its 32-element chunk conflict-free: chunk c of token t is
// four 16-byte quarters at xs + ((t * 4 + v) * NC + c) * 16 bytes, v < 4.
// sX[t * NC + c] is the chunk's sum.
__device__ __noinline__ void fx_stage_x(const uint16_t* x, const float* resid,
                                        const float* denom, int T, int H, uint16_t* xs,
                                        float* sX, int ct) {
    const int NC = H >> 5;
    uint4* xq = reinterpret_cast<uint4*>(xs);
#pragma unroll 1
    for (int i = ct; i < T * NC; i += NCT) {
        const int t = i / NC, c = i - t * NC;
        float sum = 0.0f;
        if (x != nullptr) {
            const uint4* p = reinterpret_cast<const uint4*>(x + size_t(t) * H + 32 * c);
            uint4 u[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) u[v] = __ldg(p + v);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint32_t wv[4] = {u[v].x, u[v].y, u[v].z, u[v].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) sum += bf16_lo(wv[j]) + bf16_hi(wv[j]);
                xq[(size_t(t) * 4 + v) * NC + c] = u[v];
            }
        } else {
            // bf16(r / denom): 8 elements (one 16-byte quarter) at a time
            const float* r = resid + size_t(t) * H + 32 * c;
            const float d = denom[t];
#pragma unroll 1
            for (int v = 0; v < 4; ++v) {
                const float4 f0 = ldcg_f4(r + 8 * v), f1 = ldcg_f4(r + 8 * v + 4);
                const uint32_t w0 = uint32_t(f32_to_bf16(f0.x / d)) |
                                    (uint32_t(f32_to_bf16(f0.y / d)) << 16);
                const uint32_t w1 = uint32_t(f32_to_bf16(f0.z / d)) |
                                    (uint32_t(f32_to_bf16(f0.w / d)) << 16);
                const uint32_t w2 = uint32_t(f32_to_bf16(f1.x / d)) |
                                    (uint32_t(f32_to_bf16(f1.y / d)) << 16);
                const uint32_t w3 = uint32_t(f32_to_bf16(f1.z / d)) |
                                    (uint32_t(f32_to_bf16(f1.w / d)) << 16);
                sum += bf16_lo(w0) + bf16_hi(w0);
                sum += bf16_lo(w1) + bf16_hi(w1);
                sum += bf16_lo(w2) + bf16_hi(w2);
                sum += bf16_lo(w3) + bf16_hi(w3);
                xq[(size_t(t) * 4 + v) * NC + c] = make_uint4(w0, w1, w2, w3);
            }
        }
        sX[i] = sum;
    }
}

// Token t's activations as fp32 pairs for lane-owned chunks c = lane + 32 m.
template <int MC>
__device__ __forceinline__ void xs_load(const uint16_t* xs, const float* sX, int t, int NC,
                                        int lane, uint64_t (&x2)[MC][16], float (&X)[MC]) {
    const uint4* xq = reinterpret_cast<const uint4*>(xs);
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        if (c < NC) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = xq[(size_t(t) * 4 + v) * NC + c];
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) x2[m][4 * v + i] = pk(bf16_lo(wv[i]), bf16_hi(wv[i]));
            }
            X[m] = sX[size_t(t) * NC + c];
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) x2[m][j] = 0ull;
            X[m] = 0.0f;
        }
    }
}

// --------------------------------------------------------- dot products
// One bf16 router row (in shared memory) . x: the warp's sum.
template <int MC>
__device__ __forceinline__ float router_dot(const uint8_t* row, const uint64_t (&x2)[MC][16],
                                            int NC, int lane) {
    uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        if (c < NC) {
            const uint4* wp = reinterpret_cast<const uint4*>(row + 64 * c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 w = wp[v];
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t f = pk(bf16_lo(ww[i]), bf16_hi(ww[i]));
                    if (i & 1)
                        acc1 = ffma2(f, x2[m][4 * v + i], acc1);
                    else
                        acc0 = ffma2(f, x2[m][4 * v + i], acc0);
                }
            }
        }
    }
    const float2 a0 = upk(acc0), a1 = upk(acc1);
    return warp_sum((a0.x + a0.y) + (a1.x + a1.y));
}

// Gate and up products of row pair pp of a chunk (packed rows at sq, scales
// at ss): the warp's sums.
template <int MC>
__device__ __forceinline__ void pair_dot(const uint8_t* sq, const uint16_t* ss, int pp, int H,
                                         const uint64_t (&x2)[MC][16], const float (&X)[MC],
                                         int NC, int lane, float& g, float& u) {
    const size_t qrow = size_t(H) >> 1, srow = size_t(H) >> 5;
    float acc[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const uint8_t* qr = sq + size_t(2 * pp + r) * qrow;
        const uint16_t* sr = ss + size_t(2 * pp + r) * srow;
        float v = 0.0f;
#pragma unroll
        for (int m = 0; m < MC; ++m) {
            const int c = lane + 32 * m;
            if (c < NC) {
                const uint4 q = *reinterpret_cast<const uint4*>(qr + 16 * c);
                v += group_dot(dot_chunk(q, x2[m]), X[m], f16_to_f32(sr[c]));
            }
        }
        acc[r] = warp_sum(v);
    }
    g = acc[0];
    u = acc[1];
}

// ------------------------------------------------------------- phase A/B
// Router rows [ra0, ra1) in chunks of rr rows -> logits[t][e] (+ bias).
template <int MC>
__device__ __noinline__ uint32_t fx_router(Ring R, uint32_t k, int ra0, int ra1, int rr,
                                           const float* bias, int E, float* logits,
                                           const uint16_t* xs, const float* sX, int T, int H,
                                           int cw, int lane) {
    const int NC = H >> 5;
    uint64_t x2[MC][16];
    float X[MC];
    int xt = -1;
    #pragma unroll 1
    for (int r = ra0; r < ra1; r += rr, ++k) {
        const int nr = min(rr, ra1 - r);
        const uint8_t* sl = ring_wait(R, k, lane);
        #pragma unroll 1
        for (int it = cw; it < nr * T; it += NW) {
            const int rw = it / T, t = it - rw * T, e = r + rw;
            if (t != xt) {
                xs_load<MC>(xs, sX, t, NC, lane, x2, X);
                xt = t;
            }
            const float v = router_dot<MC>(sl + size_t(rw) * 2 * H, x2, NC, lane);
            if (lane == 0)
                logits[size_t(t) * (E + 1) + e] =
                    v + ((e < E && bias != nullptr) ? __ldg(bias + e) : 0.0f);
        }
        ring_release(R, k, lane);
    }
    return k;
}

// Gate/up row pairs [rp0, rp1) of experts with Iu pairs each (pair rp is
// pair rp % Iu of expert rp / Iu), in chunks of at most pb pairs within one
// expert.  Expert j's slots are off[j] .. off[j] + cnt[j] - 1 and tok[s] is
// slot s's token (tok NULL: slot s is token s).  dst[s * Iu + i] =
// silu(gate_i) * up_i.  first: stamp of the first chunk's arrival, or NULL.
template <int MC>
__device__ __noinline__ uint32_t fx_gate_up(Ring R, uint32_t k, long long rp0, long long rp1,
                                            int Iu, int pb, int stage_q, const int* off,
                                            const int* cnt, const int* tok, float* dst,
                                            const uint16_t* xs, const float* sX, int T, int H,
                                            int cw, int lane, unsigned long long* first) {
    const int NC = H >> 5;
    uint64_t x2[MC][16];
    float X[MC];
    int xt = -1;
    #pragma unroll 1
    for (long long rp = rp0; rp < rp1; ++k) {
        const int j = int(rp / Iu), i0 = int(rp % Iu);
        const int nb = int(min((long long)pb, min((long long)(Iu - i0), rp1 - rp)));
        const uint8_t* sl = ring_wait(R, k, lane);
        if (first != nullptr && rp == rp0) *first = global_clock();
        const uint16_t* ss = reinterpret_cast<const uint16_t*>(sl + stage_q);
        const int s0 = off[j], sc = cnt[j];
        #pragma unroll 1
        for (int pp = cw; pp < nb; pp += NW) {
            #pragma unroll 1
            for (int si = 0; si < sc; ++si) {
                const int s = s0 + si;
                const int t = tok != nullptr ? tok[s] : s;
                if (t < 0 || t >= T) continue;
                if (t != xt) {
                    xs_load<MC>(xs, sX, t, NC, lane, x2, X);
                    xt = t;
                }
                float g, u;
                pair_dot<MC>(sl, ss, pp, H, x2, X, NC, lane, g, u);
                if (lane == 0) dst[size_t(s) * Iu + i0 + pp] = silu_mul(g, u);
            }
        }
        ring_release(R, k, lane);
        rp += nb;
    }
    return k;
}

// --------------------------------------------------------------- phase C
// The down phase walks units -- u = 0 the shared expert (its T tokens are
// its slots), u >= 1 the touched experts in ascending id -- and packs them
// into chunks: an item is a unit's down rows for this CTA's output rows
// (nrow rows of L/2 packed bytes and L/32 scales) followed by the SwiGLU
// vectors (L floats each) of ns of its slots.  A unit whose slots do not fit
// is split over several items (its rows copied again).  The producer and
// the consumers run the same packing.
struct CItem {
    int u, s0, ns, woff, hoff;
};
struct CPack {
    int u, sdone;
};

__device__ __forceinline__ uint32_t unit_wbytes(int nrow, int L) {
    return (uint32_t(nrow) * uint32_t((L >> 1) + (L >> 4)) + 15u) & ~15u;
}

__device__ __noinline__ int fx_c_chunk(CPack& it, int nunits, const int* cnt, int T, int I,
                                       int Is, int nrow, uint32_t SB, CItem* items) {
    int n = 0;
    uint32_t bytes = 0;
    while (it.u < nunits && n < kFxMaxItems) {
        const bool sh = it.u == 0;
        const int L = sh ? Is : I;
        const int cu = sh ? T : cnt[it.u - 1];
        const uint32_t wb = unit_wbytes(nrow, L), hb = uint32_t(L) * 4u;
        if (bytes + wb + hb > SB) break;
        const int fit = int((SB - bytes - wb) / hb);
        const int ns = min(cu - it.sdone, fit);
        items[n].u = it.u;
        items[n].s0 = it.sdone;
        items[n].ns = ns;
        items[n].woff = int(bytes);
        items[n].hoff = int(bytes + wb);
        ++n;
        bytes += wb + uint32_t(ns) * hb;
        it.sdone += ns;
        if (it.sdone >= cu) {
            ++it.u;
            it.sdone = 0;
        }
    }
    return n;
}

// One item: s_y[(ybase + si) * ldy + row] = sum_i h[si][i] W[row][i] for its
// ns slots, weights and SwiGLU vectors in shared memory.  Lane (rs, c) holds
// chunk c of rows rs, rs + RPW, ...; MR rows a lane at a time.
template <int MR>
__device__ __forceinline__ void fx_down_item(const uint8_t* sq, const uint16_t* ss, int L,
                                             int nrow, int lane, const float* hb, int ns,
                                             float* s_y, int ybase, int ldy) {
    const int NCd = L >> 5, RPW = 32 / NCd;
    const int c = lane & (NCd - 1), rs = lane / NCd;
    const int npass = (nrow + RPW - 1) / RPW;          // uniform over the warp
    const size_t qrow = size_t(L) >> 1, srow = size_t(L) >> 5;
    #pragma unroll 1
    for (int si = 0; si < ns; ++si) {
        const float* hp = hb + size_t(si) * L + 32 * c;
        uint64_t x2[16];
        float X = 0.0f;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = *reinterpret_cast<const float4*>(hp + 4 * v);
            x2[2 * v] = pk(f.x, f.y);
            x2[2 * v + 1] = pk(f.z, f.w);
            X += (f.x + f.y) + (f.z + f.w);
        }
        #pragma unroll 1
        for (int pg = 0; pg < npass; pg += MR) {
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                if (pg + m < npass) {
                    const int row = rs + (pg + m) * RPW;
                    float part = 0.0f;
                    if (row < nrow) {
                        const uint4 q = *reinterpret_cast<const uint4*>(sq + row * qrow + 16 * c);
                        part = group_dot(dot_chunk(q, x2), X, f16_to_f32(ss[row * srow + c]));
                    }
                    part = group_sum(part, NCd);
                    if (c == 0 && row < nrow) s_y[size_t(ybase + si) * ldy + row] = part;
                }
            }
        }
    }
}

template <int MR>
__device__ __noinline__ uint32_t fx_down(Ring R, uint32_t k, int nunits, const int* off,
                                         const int* cnt, int T, int TK, int I, int Is, int nrow,
                                         float* s_y, int cw, int lane) {
    CPack it{0, 0};
    CItem items[kFxMaxItems];
    int gi = 0;
    #pragma unroll 1
    for (;; ++k) {
        const int n = fx_c_chunk(it, nunits, cnt, T, I, Is, nrow, R.SB, items);
        if (n == 0) break;
        const uint8_t* sl = ring_wait(R, k, lane);
        #pragma unroll 1
        for (int i = 0; i < n; ++i, ++gi) {
            if (gi % NW != cw) continue;
            const CItem& c = items[i];
            const bool sh = c.u == 0;
            const int L = sh ? Is : I;
            const uint8_t* sq = sl + c.woff;
            const uint16_t* ss = reinterpret_cast<const uint16_t*>(sq + size_t(nrow) * (L >> 1));
            const float* hb = reinterpret_cast<const float*>(sl + c.hoff);
            const int ybase = sh ? TK + c.s0 : off[c.u - 1] + c.s0;
            fx_down_item<MR>(sq, ss, L, nrow, lane, hb, c.ns, s_y, ybase, nrow);
        }
        ring_release(R, k, lane);
    }
    return k;
}

// ---------------------------------------------------- routing and combine
__device__ __noinline__ void fx_route(const float* logits, int T, int E, int K,
                                      const int32_t* forced_ids, const float* forced_w,
                                      int* s_ids, float* s_w, float* s_sig, float* scratch,
                                      uint32_t* err, int ct, SPlan* P, int* s_cnt, int* s_off,
                                      int* s_wsum, int* s_inv) {
    route_cta(logits, T, E, K, forced_ids, forced_w, s_ids, s_w, s_sig, scratch, err, ct, NCT,
              ConsSync{});
    const BucketOut none{nullptr, nullptr, nullptr, nullptr, nullptr};
    bucket_cta(s_ids, T, K, E, s_cnt, s_off, s_wsum, *P, s_inv, none, ct, NCT, ConsSync{});
}

// out[t][o] = bf16( sum_{k ascending} w[t][k] y[inv[t*K+k]][o] + sig[t] S[t][o] )
// for this CTA's rows; resid (optional) += the bf16 output, kept in s_rn.
__device__ __noinline__ void fx_combine(const float* s_y, const int* s_inv, const float* s_w,
                                        const float* s_sig, int T, int K, int TK, int H, int o0,
                                        int nrow, uint16_t* out, float* resid, float* s_rn,
                                        int ct) {
    #pragma unroll 1
    for (int i = ct; i < T * nrow; i += NCT) {
        const int t = i / nrow, r = i - t * nrow, o = o0 + r;
        float acc = 0.0f;
        #pragma unroll 1
        for (int kk = 0; kk < K; ++kk) {
            const int sl = s_inv[t * K + kk];
            if (sl < 0 || sl >= TK) continue;
            acc += s_w[t * K + kk] * s_y[size_t(sl) * nrow + r];
        }
        const float v = acc + s_sig[t] * s_y[size_t(TK + t) * nrow + r];
        const uint16_t ob = f32_to_bf16(v);
        if (out != nullptr) out[size_t(t) * H + o] = ob;
        if (resid != nullptr) {
            float* rp = resid + size_t(t) * H + o;
            const float rn = __ldcg(rp) + bf16_lo(uint32_t(ob));
            *rp = rn;
            s_rn[size_t(t) * nrow + r] = rn;
        }
    }
}

// RMSNorm denominators of the layer's input: from the residual itself at
// the first layer, else from the previous layer's per-CTA partial sums of
// squares (summed in a fixed order: the same result in every CTA).
__device__ __noinline__ void fx_denominators(const float* resid, const float* ssq, int first,
                                             int T, int H, int G, float eps, float* s_denom,
                                             int cw, int lane) {
    #pragma unroll 1
    for (int t = cw; t < T; t += NW) {
        float ss = 0.0f;
        if (first) {
            const float* rt = resid + size_t(t) * H;
            #pragma unroll 1
            for (int h = lane * 4; h < H; h += 128) {
                const float4 v = ldcg_f4(rt + h);
                ss += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
            }
        } else {
            #pragma unroll 1
            for (int b = lane; b < G; b += 32) ss += __ldcg(ssq + size_t(b) * T + t);
        }
        ss = warp_sum(ss);
        if (lane == 0) s_denom[t] = sqrtf(ss / float(H) + eps);
    }
}

// ---------------------------------------------------------------- kernel
template <int MC, int MR>
__global__ void __launch_bounds__(kFxThreads, 1) k_moe_decode(const __grid_constant__ FusedLaunch a) {
    extern __shared__ __align__(128) uint8_t fx_dyn[];
    __shared__ SPlan P;
    __shared__ int s_ids[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_w[kDecodeMaxTokens * kMaxTopK];
    __shared__ int s_inv[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_sig[kDecodeMaxTokens];
    __shared__ float s_denom[kDecodeMaxTokens];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_wsum[32];
    __shared__ int s_shared_slots[2];                 // the shared expert: offset 0, T slots
    __shared__ __align__(8) uint64_t full[kFxMaxSlots], empty[kFxMaxSlots];
    __shared__ __align__(8) uint64_t plan_bar, h_bar;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int T = a.T, H = a.H, E = a.E, K = a.K, I = a.I, Is = a.Is, TK = T * K;
    const int G = gridDim.x, cta = blockIdx.x;
    const int NC = H >> 5;
    // chunk trace of CTA 0 (profiling): the producer thread and consumer warp 0
    unsigned long long* trace =
        (a.stamps != nullptr && cta == 0 && (tid == 0 || tid == 32))
            ? a.stamps + size_t(kFxMaxGrid) * kFxStampsPerLayer
            : nullptr;
    const Ring R{fx_dyn, full, empty, uint32_t(a.slots), uint32_t(a.slot_bytes), a.err, trace};
    uint16_t* xs = reinterpret_cast<uint16_t*>(fx_dyn + size_t(a.slots) * a.slot_bytes);
    float* sX = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + size_t(T) * H * 2);
    float* scratch = sX + size_t(T) * NC;

    // this CTA's static shares: router rows, shared gate/up pairs, output rows
    const bool forced = a.forced_ids != nullptr;
    const int rbase = forced ? E : 0, NR = E + 1 - rbase;
    const int ra0 = rbase + int((long long)cta * NR / G);
    const int ra1 = rbase + int((long long)(cta + 1) * NR / G);
    const int pa0 = int((long long)cta * Is / G), pa1 = int((long long)(cta + 1) * Is / G);
    const int og = a.og, nog = H / og;
    const int o0 = og * int((long long)cta * nog / G);
    const int nrow = og * int((long long)(cta + 1) * nog / G) - o0;

    if (tid == 0) {
        if (a.stamps != nullptr) a.stamps[size_t(cta) * kFxStampsPerLayer + 9] = global_clock();
        #pragma unroll 1
        for (int i = 0; i < a.slots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kFxConsumers);
        }
        mbar_init(&plan_bar, 1);
        mbar_init(&h_bar, 1);
        mbar_fence_init();
        s_shared_slots[0] = 0;
        s_shared_slots[1] = T;
    }
    __syncthreads();

    if (wid == 0) {
        // ---------------------------------------------------------- producer
        if (lane != 0) return;
        uint32_t k = 0;
        auto issue_pairs = [&](uint32_t kk, const uint8_t* q, const uint16_t* sc, int i0, int nb) {
            uint8_t* dst = ring_acquire(R, kk);
            uint64_t* fb = &full[kk % R.S];
            const uint32_t bq = uint32_t(nb) * uint32_t(H);
            const uint32_t bs = uint32_t(nb) * uint32_t(H >> 3);
            mbar_expect_tx(fb, bq + bs);
            bulk_g2s(dst, q + size_t(2 * i0) * (H >> 1), bq, fb);
            bulk_g2s(dst + a.stage_q, sc + size_t(2 * i0) * (H >> 5), bs, fb);
        };
        CItem items[kFxMaxItems];
        #pragma unroll 1
        for (int l = 0; l < a.n_layers; ++l) {
            const strata_moe_layer& L = a.layers[l];
            const uint16_t* router = static_cast<const uint16_t*>(L.router_dev);
            #pragma unroll 1
            for (int r = ra0; r < ra1; r += a.rr, ++k) {
                const int nr = min(a.rr, ra1 - r);
                uint8_t* dst = ring_acquire(R, k);
                uint64_t* fb = &full[k % R.S];
                const uint32_t bytes = uint32_t(nr) * 2u * uint32_t(H);
                mbar_expect_tx(fb, bytes);
                bulk_g2s(dst, router + size_t(r) * H, bytes, fb);
            }
            #pragma unroll 1
            for (int p = pa0; p < pa1; p += a.pb, ++k)
                issue_pairs(k, L.sh_gu_q_dev, L.sh_gu_s_dev, p, min(a.pb, pa1 - p));
            // the routed chunks need this layer's plan
            if (!fx_wait(&plan_bar, uint32_t(l) & 1u, a.err)) latch_timeout(a.err, 22, 0, l, 0);
            const int n_exp = P.n;
            const long long RP = (long long)n_exp * I;
            const long long b0 = (long long)cta * RP / G, b1 = (long long)(cta + 1) * RP / G;
            #pragma unroll 1
            for (long long rp = b0; rp < b1; ++k) {
                const int j = int(rp / I), i0 = int(rp % I);
                const int nb = int(min((long long)a.pb, min((long long)(I - i0), b1 - rp)));
                const size_t e = size_t(P.e[j]);
                issue_pairs(k, L.gu_q_dev + e * 2 * I * (H >> 1),
                            L.gu_s_dev + e * 2 * I * (H >> 5), i0, nb);
                rp += nb;
            }
            if (nrow <= 0) continue;
            // Down chunks.  Their weights first, without arriving: the first
            // S of them take slots last used by chunks that need nothing
            // more from this thread, so waiting for those slots is safe.
            // The SwiGLU vectors exist once the consumers pass the second
            // barrier (h_bar); then every chunk gets them and its arrival.
            const int nunits = 1 + n_exp;
            const uint32_t kc0 = k;
            auto unit_src = [&](int u, int L_, const uint8_t*& q, const uint16_t*& sc) {
                const bool sh = u == 0;
                const size_t e = sh ? 0 : size_t(P.e[u - 1]);
                q = sh ? L.sh_dn_q_dev : L.dn_q_dev + e * H * (L_ >> 1);
                sc = sh ? L.sh_dn_s_dev : L.dn_s_dev + e * H * (L_ >> 5);
            };
            auto issue_weights = [&](uint8_t* dst, uint64_t* fb, const CItem* it, int n) {
                #pragma unroll 1
                for (int i = 0; i < n; ++i) {
                    const int Lu = it[i].u == 0 ? Is : I;
                    const uint8_t* q;
                    const uint16_t* sc;
                    unit_src(it[i].u, Lu, q, sc);
                    const uint32_t bq = uint32_t(nrow) * uint32_t(Lu >> 1);
                    bulk_g2s(dst + it[i].woff, q + size_t(o0) * (Lu >> 1), bq, fb);
                    bulk_g2s(dst + it[i].woff + bq, sc + size_t(o0) * (Lu >> 5),
                             uint32_t(nrow) * uint32_t(Lu >> 4), fb);
                }
            };
            auto issue_h = [&](uint8_t* dst, uint64_t* fb, const CItem* it, int n) {
                #pragma unroll 1
                for (int i = 0; i < n; ++i) {
                    const bool sh = it[i].u == 0;
                    const int Lu = sh ? Is : I;
                    const float* src = sh ? a.hs + size_t(it[i].s0) * Is
                                          : a.h + size_t(P.off[it[i].u - 1] + it[i].s0) * I;
                    bulk_g2s(dst + it[i].hoff, src, uint32_t(it[i].ns) * uint32_t(Lu) * 4u, fb);
                }
            };
            auto chunk_bytes = [&](const CItem* it, int n, uint32_t& wbytes, uint32_t& hbytes) {
                wbytes = 0;
                hbytes = 0;
                #pragma unroll 1
                for (int i = 0; i < n; ++i) {
                    const int Lu = it[i].u == 0 ? Is : I;
                    wbytes += uint32_t(nrow) * uint32_t((Lu >> 1) + (Lu >> 4));
                    hbytes += uint32_t(it[i].ns) * uint32_t(Lu) * 4u;
                }
            };
            CPack pk1{0, 0};
            uint32_t nw = 0;
            #pragma unroll 1
            for (; nw < R.S; ++nw) {
                const int n = fx_c_chunk(pk1, nunits, P.cnt, T, I, Is, nrow, R.SB, items);
                if (n == 0) break;
                uint8_t* dst = ring_acquire(R, kc0 + nw);
                uint64_t* fb = &full[(kc0 + nw) % R.S];
                uint32_t wb, hb;
                chunk_bytes(items, n, wb, hb);
                mbar_expect_tx_only(fb, wb);
                issue_weights(dst, fb, items, n);
            }
            if (!fx_wait(&h_bar, uint32_t(l) & 1u, a.err)) latch_timeout(a.err, 24, 0, l, 0);
            fence_proxy_async_global();
            CPack pk2{0, 0};
            #pragma unroll 1
            for (uint32_t c = 0;; ++c) {
                const int n = fx_c_chunk(pk2, nunits, P.cnt, T, I, Is, nrow, R.SB, items);
                if (n == 0) break;
                uint32_t wb, hb;
                chunk_bytes(items, n, wb, hb);
                if (c < nw) {
                    uint8_t* dst = R.base + size_t((kc0 + c) % R.S) * R.SB;
                    uint64_t* fb = &full[(kc0 + c) % R.S];
                    mbar_expect_tx(fb, hb);
                    issue_h(dst, fb, items, n);
                    if (R.trace != nullptr && kc0 + c < kFxTraceChunks)
                        R.trace[3 * kFxTraceChunks + kc0 + c] = global_clock();
                } else {
                    uint8_t* dst = ring_acquire(R, kc0 + c);
                    uint64_t* fb = &full[(kc0 + c) % R.S];
                    mbar_expect_tx(fb, wb + hb);
                    issue_weights(dst, fb, items, n);
                    issue_h(dst, fb, items, n);
                }
                ++k;
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int ct = tid - 32, cw = wid - 1;
    const bool stamp = a.stamps != nullptr && ct == 0;     // first layer, every CTA
    float* s_y = scratch;                                   // [(TK + T)][nrow]
    float* s_rn = scratch + size_t(TK + T) * (nrow > 0 ? nrow : 1);   // [T][nrow]
    uint32_t k = 0;

    #pragma unroll 1
    for (int l = 0; l < a.n_layers; ++l) {
        const strata_moe_layer& L = a.layers[l];
        unsigned long long* st =
            (stamp && l == 0) ? a.stamps + size_t(cta) * kFxStampsPerLayer : nullptr;
        if (st) st[0] = global_clock();
        if (a.x == nullptr) {
            fx_denominators(a.resid, a.ssq, l == 0, T, H, G, a.eps, s_denom, cw, lane);
            ConsSync{}();
            if (l == 0 && a.x_out != nullptr)
                #pragma unroll 1
                for (int i = ct; i < T * nrow; i += NCT) {
                    const int t = i / nrow, o = o0 + i % nrow;
                    a.x_out[size_t(t) * H + o] =
                        f32_to_bf16(__ldcg(a.resid + size_t(t) * H + o) / s_denom[t]);
                }
        }
        fx_stage_x(a.x, a.resid, s_denom, T, H, xs, sX, ct);
        ConsSync{}();

        // ---- A: router rows -> logits; shared gate/up pairs -> hs
        k = fx_router<MC>(R, k, ra0, ra1, a.rr, L.router_bias_dev, E, a.logits, xs, sX, T, H,
                          cw, lane);
        k = fx_gate_up<MC>(R, k, pa0, pa1, Is, a.pb, a.stage_q, s_shared_slots,
                           s_shared_slots + 1, nullptr, a.hs, xs, sX, T, H, cw, lane, nullptr);
        fence_proxy_async_global();
        if (st) st[1] = global_clock();
        fx_grid_sync(a.bar, a.err, ct, 31, l);
        if (st) st[2] = global_clock();

        // ---- B: routing (every CTA alike), then the routed gate/up pairs
        fx_route(a.logits, T, E, K, forced ? a.forced_ids + size_t(l) * TK : nullptr,
                 forced ? a.forced_w + size_t(l) * TK : nullptr, s_ids, s_w, s_sig, scratch,
                 a.err, ct, &P, s_cnt, s_off, s_wsum, s_inv);
        if (ct == 0) mbar_arrive(&plan_bar);
        if (st) st[10] = global_clock();
        if (cta == 0 && l == 0) {
            #pragma unroll 1
            for (int p = ct; p < TK; p += NCT) {
                if (a.ids_user) a.ids_user[p] = s_ids[p];
                if (a.w_user) a.w_user[p] = s_w[p];
            }
            if (a.sig_user)
                #pragma unroll 1
                for (int t = ct; t < T; t += NCT) a.sig_user[t] = s_sig[t];
        }
        if (st) st[3] = global_clock();
        const long long RP = (long long)P.n * I;
        const long long b0 = (long long)cta * RP / G, b1 = (long long)(cta + 1) * RP / G;
        if (st) st[8] = global_clock();
        k = fx_gate_up<MC>(R, k, b0, b1, I, a.pb, a.stage_q, P.off, P.cnt, P.tok, a.h, xs, sX,
                           T, H, cw, lane, st ? st + 8 : nullptr);
        fence_proxy_async_global();
        if (st) st[4] = global_clock();
        fx_grid_sync(a.bar, a.err, ct, 32, l);
        if (ct == 0) mbar_arrive(&h_bar);
        if (st) st[5] = global_clock();

        // ---- C: down rows of every unit for this CTA's output rows, combine
        if (nrow > 0) {
            #pragma unroll 1
            for (int i = ct; i < (TK + T) * nrow; i += NCT) s_y[i] = 0.0f;
            ConsSync{}();
            if (st) st[11] = global_clock();
            k = fx_down<MR>(R, k, 1 + P.n, P.off, P.cnt, T, TK, I, Is, nrow, s_y, cw, lane);
            if (st) st[13] = global_clock();
            ConsSync{}();
            if (st) st[6] = global_clock();
            fx_combine(s_y, s_inv, s_w, s_sig, T, K, TK, H, o0, nrow,
                       l + 1 == a.n_layers ? a.out : nullptr, a.resid, s_rn, ct);
        } else if (st) {
            st[11] = st[13] = st[6] = global_clock();
        }
        if (a.resid != nullptr && l + 1 < a.n_layers) {
            // partial sums of squares of this CTA's rows of the new residual
            ConsSync{}();
            #pragma unroll 1
            for (int t = cw; t < T; t += NW) {
                float v = 0.0f;
                #pragma unroll 1
                for (int r = lane; r < nrow; r += 32) {
                    const float x = s_rn[size_t(t) * nrow + r];
                    v += x * x;
                }
                v = warp_sum(v);
                if (lane == 0) a.ssq[size_t(cta) * T + t] = v;
            }
            fx_grid_sync(a.bar, a.err, ct, 33, l);
        }
        if (st) st[7] = global_clock();
    }
    // Every chunk was waited for above; after a wait that ran out, make sure
    // no copy into this CTA's shared memory is still in flight at exit.
    if (ct == 0 && *reinterpret_cast<const volatile uint32_t*>(a.err) == 4u) {
        #pragma unroll 1
        for (uint32_t slot = 0; slot < uint32_t(a.slots) && slot < k; ++slot) {
            const uint32_t last = slot + ((k - 1 - slot) / a.slots) * a.slots;
            #pragma unroll 1
            for (uint32_t i = 0; i < kWaitLimit; ++i)
                if (mbar_try_wait(&full[slot], (last / a.slots) & 1)) break;
        }
    }
}

// ------------------------------------------------------------------ host
namespace {

// Per kernel instantiation and device: its static shared memory, the
// device's opt-in limit, and the largest dynamic size already allowed (and
// checked for one resident CTA per SM).
struct FxDevCache {
    int known = 0, optin = 0;
    size_t static_smem = 0, dyn_ok = 0;
};
constexpr int kFxCacheDevices = 64;
template <int MC, int MR>
FxDevCache* fx_cache(int dev) {
    static FxDevCache c[kFxCacheDevices];
    return (dev >= 0 && dev < kFxCacheDevices) ? &c[dev] : nullptr;
}
std::mutex g_fx_mu;

template <int MC, int MR>
cudaError_t launch_fx(FusedLaunch& a, int grid, cudaStream_t s) {
    auto kernel = k_moe_decode<MC, MR>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_fx_mu);
    FxDevCache tmp;
    FxDevCache* cache = fx_cache<MC, MR>(dev);
    if (cache == nullptr) cache = &tmp;
    if (!cache->known) {
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, kernel)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&cache->optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        dev)) != cudaSuccess)
            return e;
        cache->static_smem = fa.sharedSizeBytes;
        cache->known = 1;
    }
    // after the ring: the staged activations (bf16) and their chunk sums,
    // then scratch for the selection's per-warp logits or for the down
    // products and the new residual rows (never live at the same time)
    const int nog = a.H / a.og;
    const int nrow_max = a.og * ((nog + grid - 1) / grid);
    const int TK = a.T * a.K;
    const size_t xbytes = size_t(a.T) * a.H * 2 + size_t(a.T) * (a.H / 32) * sizeof(float);
    const size_t sel = size_t(kFxConsumers) * (a.E + 16) * sizeof(float);
    const size_t dn = size_t(TK + 2 * a.T) * (nrow_max > 0 ? nrow_max : 1) * sizeof(float);
    const size_t scratch = ((sel > dn ? sel : dn) + 127) & ~size_t(127);
    const long long avail = (long long)cache->optin - (long long)cache->static_smem - 1024 -
                            (long long)xbytes - (long long)scratch;
    int S = int(avail / a.slot_bytes);
    if (S > kFxMaxSlots) S = kFxMaxSlots;
    if (S < 2) return cudaErrorInvalidConfiguration;
    a.slots = S;
    const size_t dyn = size_t(S) * a.slot_bytes + xbytes + scratch;
    if (dyn > cache->dyn_ok) {
        if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(dyn))) != cudaSuccess)
            return e;
        int per_sm = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kFxThreads,
                                                               dyn)) != cudaSuccess)
            return e;
        if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
        cache->dyn_ok = dyn;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFxThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e == cudaSuccess) prof_after_launch(s);
    return e;
}

}  // namespace

cudaError_t launch_fused_decode(FusedLaunch& a, cudaStream_t s) {
    const Dev d = device_info();
    const int grid = d.sms < kFxMaxGrid ? d.sms : kFxMaxGrid;
    const int Lmin = a.I < a.Is ? a.I : a.Is, Lmax = a.I > a.Is ? a.I : a.Is;
    // output rows in multiples of og, so every unit's scale rows start on a
    // 16-byte boundary (a row of L/32 fp16 scales is L/16 bytes)
    a.og = Lmin >= 256 ? 1 : 256 / Lmin;
    const int nog = a.H / a.og;
    const int nrow_max = a.og * ((nog + grid - 1) / grid);
    a.pb = kFxPairs;
    a.stage_q = a.pb * a.H;                                   // pb pairs of packed rows
    a.slot_bytes = a.stage_q + a.pb * (a.H >> 3);             // + their scales
    // a down item needs room for its rows and at least one SwiGLU vector
    a.ub = ((nrow_max * ((Lmax >> 1) + (Lmax >> 4))) + 15) & ~15;
    if (a.ub + 4 * Lmax > a.slot_bytes) a.slot_bytes = (a.ub + 4 * Lmax + 127) & ~127;
    a.rr = a.slot_bytes / (2 * a.H);
    a.uc = 0;
    if (a.rr < 1) return cudaErrorInvalidConfiguration;
    const int mc = (a.H + 1023) / 1024;
    if (mc <= 1) return launch_fx<1, 4>(a, grid, s);
    if (mc <= 2) return launch_fx<2, 4>(a, grid, s);
    return launch_fx<4, 4>(a, grid, s);
}

}  // namespace strata
