// persist.cu -- a decode-size MoE layer, or a stack of residual MoE layers,
// as ONE persistent kernel per call: one CTA per SM, no kernel boundary and
// no grid-wide barrier between the layer's steps.
//
// PolyStrata ("Models and backends", section "What was tuned") finds decode
// launch-bound: ~35 small launches a layer and the engine waiting for the
// card at every router.  Strata ("Qwen3.6-35B-A3B: pictures, several
// requests at once and speed", section "Speed") fuses the router product,
// top-k and grouping into one launch and the MoE end into another.  Here
// the whole layer is one launch, and a stack of layers is one launch too.
//
// Per layer, in every CTA (one producer warp issuing 1-D bulk copies into
// shared memory, seven consumer warps computing):
//   R  router rows (E + 1: the last is the shared-expert gate) and the
//      shared expert's gate/up row pairs: this CTA's share, by bytes, of
//      the weights that do not depend on routing.  Its copy is requested a
//      layer ahead (the first layer's at kernel start, before waiting for
//      the previous kernel), so R computes from shared memory.
//   S  every token's top-K from all the logits, softmax weights, sigmoid
//      gate, bucketing: the same result in every CTA.
//   G  this CTA's share of the touched experts' gate/up row pairs, cut by
//      cost (tokens + 1 per row pair), streamed through a ring of stages of
//      a few row pairs, one warp a stage; SwiGLU.  The down rows this CTA
//      owns for every touched expert are requested right behind.
//   D  down products of this CTA's output rows for every touched expert and
//      the shared expert, then the fixed-order weighted combine; the stack
//      adds the bf16 output to the fp32 residual, and the next layer starts
//      with the RMSNorm of the residual in every CTA.
//
// Cross-CTA values (logits, the shared and routed SwiGLU vectors, a stack's
// residual) go through the workspace as 64-bit words: the value in the low
// half, a tag naming the exchange in the high half.  A 64-bit access is
// single-copy atomic, so a reader that sees the tag sees the value: it polls
// the data itself, one L2 round trip, with no fence and no flag.  Tags are
// the workspace's exchange count (one counter per CTA, all equal between
// launches) plus the exchange's number in the launch, so a word left by an
// earlier launch never carries the current tag.
//
// The arithmetic (int4 byte placement, per-lane partial sums, warp sums,
// SwiGLU, combine order, RMSNorm) is that of the three-kernel decode path,
// so both paths give the same bits.  Every wait is bounded: one that runs
// out latches STRATA_ETIMEOUT and the kernel runs on to its end with wrong
// values instead of hanging.

#include <math.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "route.cuh"

namespace strata {

constexpr int kPxThreads = 32 * (kPxConsumers + 1);
constexpr uint32_t kLlWaitLimit = 1u << 21;     // polls (L2 round trips): a second or two
constexpr int kPxExchanges = 3;                  // tagged exchanges a layer

static std::atomic<uint32_t> g_grid_wait_limit{0};

uint32_t grid_wait_limit() {
    const uint32_t v = g_grid_wait_limit.load(std::memory_order_relaxed);
    return v ? v : kLlWaitLimit;
}

void set_grid_wait_limit(uint32_t polls) { g_grid_wait_limit.store(polls, std::memory_order_relaxed); }

// ------------------------------------------------------------ phase trace
#ifdef STRATA_PX_TRACE
__device__ unsigned long long g_px_trace[kMaxGrid * kPxTraceSlots * kPxTracePoints];
// The global timer at phase point `pt` of layer l (of n) into this CTA's
// slot for that layer (layers 0, 1, n/2, n-1; others are not recorded).
__device__ __forceinline__ void px_trace(int l, int n, int pt) {
    const int slot = l == 0 ? 0 : l == 1 ? 1 : l == n / 2 ? 2 : l == n - 1 ? 3 : -1;
    if (slot < 0) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_px_trace[(size_t(blockIdx.x) * kPxTraceSlots + slot) * kPxTracePoints + pt] = t;
}
#else
__device__ __forceinline__ void px_trace(int, int, int) {}
#endif

// ------------------------------------------------------------ primitives
__device__ __forceinline__ void px_cbar() {   // the consumer warps only
    asm volatile("bar.sync 1, %0;" ::"r"(kPxConsumers * 32) : "memory");
}
struct PxSync {
    __device__ void operator()() const { px_cbar(); }
};
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void px_fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// try_wait with a suspend-time hint: a waiting warp sleeps (up to the hint,
// or until the phase completes) instead of spinning on the issue slots its
// sub-partition's working warps need.
__device__ __forceinline__ bool px_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// A wait that gives up at once when another wait already latched a timeout.
__device__ __forceinline__ bool px_wait(uint64_t* bar, uint32_t parity, const uint32_t* err) {
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (px_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u && ld_relaxed_u32(err) == uint32_t(STRATA_ETIMEOUT)) return false;
    }
    return false;
}

// Between two polls of a word that was not there yet: nothing.  A poll is an
// L2 round trip, which paces it; a sleep of 32 or 128 ns here measured 0.4
// and 4 us slower a layer in the 40-layer stack, the same in one layer.
__device__ __forceinline__ void px_backoff() {}

// --------------------------------------------------- tagged 64-bit words
__device__ __forceinline__ void ll_put(uint64_t* p, float v, uint32_t tag) {
    const uint64_t w = (uint64_t(tag) << 32) | uint64_t(__float_as_uint(v));
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// (no memory clobber: a poll's loads may all be in flight at once)
__device__ __forceinline__ uint64_t ll_ld(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void ll_ld2(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}
__device__ __forceinline__ bool ll_has(uint64_t w, uint32_t tag) { return uint32_t(w >> 32) == tag; }
__device__ __forceinline__ float ll_val(uint64_t w) { return __uint_as_float(uint32_t(w)); }

// The N (even) tagged words at p (16-byte aligned) into v, waiting until
// every one carries `tag`: each poll issues all N loads, then checks them.
// false: the wait ran out (v then holds whatever was read).
template <int N>
__device__ __forceinline__ bool ll_wait(const uint64_t* p, uint32_t tag, float (&v)[N],
                                        uint32_t limit, const uint32_t* err) {
    static_assert(N % 2 == 0, "pairs of words");
    for (uint32_t it = 0; it < limit; ++it) {
        uint64_t w[N];
#pragma unroll
        for (int j = 0; j < N / 2; ++j) ll_ld2(p + 2 * j, w[2 * j], w[2 * j + 1]);
        bool ok = true;
#pragma unroll
        for (int j = 0; j < N; ++j) {
            ok &= ll_has(w[j], tag);
            v[j] = ll_val(w[j]);
        }
        if (ok) return true;
        if ((it & 255u) == 255u && ld_relaxed_u32(err) == uint32_t(STRATA_ETIMEOUT)) return false;
        px_backoff();
    }
    return false;
}

// This CTA's share of the routing-independent rows: router rows [r0, r0+nr)
// of the nR requested (all E + 1, or only the gate row E under forced
// routing) and shared gate/up row pairs [p0, p0+np).  The rows are laid end
// to end by bytes and cut into G equal byte ranges; a row belongs to the
// CTA whose range holds its first byte.
struct RShare {
    int r0, nr, p0, np;
};
__host__ __device__ inline long long px_cdiv0(long long x, long long y) {
    return x <= 0 ? 0LL : (x + y - 1) / y;
}
__host__ __device__ inline long long px_min(long long x, long long y) { return x < y ? x : y; }
__host__ __device__ inline RShare px_r_share(int b, int G, int nR, int Is, int H) {
    const long long Rrow = 2LL * H, Spair = (long long)H + H / 8;
    const long long Rtot = nR * Rrow, tot = Rtot + (long long)Is * Spair;
    const long long lo = tot * b / G, hi = tot * (b + 1) / G;
    const int r0 = int(px_min(nR, px_cdiv0(lo, Rrow))), r1 = int(px_min(nR, px_cdiv0(hi, Rrow)));
    const int p0 = int(px_min(Is, px_cdiv0(lo - Rtot, Spair)));
    const int p1 = int(px_min(Is, px_cdiv0(hi - Rtot, Spair)));
    return RShare{r0, r1 - r0, p0, p1 - p0};
}

// Row pair `x` (in cost units) of the touched experts' gate/up: a row pair
// of expert j costs its tokens plus one (the read of its rows).  Returns the
// global row pair j * I + i.
__device__ inline int px_rp_at(const SPlan& P, int I, int x) {
    int cum = 0;
    for (int j = 0; j < P.n; ++j) {
        const int w = P.cnt[j] + 1, cj = w * I;
        if (x < cum + cj) return j * I + (x - cum) / w;
        cum += cj;
    }
    return P.n * I;
}
// This CTA's share of the touched experts' row pairs: it starts at row pair
// i0 of touched expert j and counts n row pairs.
struct GRange {
    int j, i0, n;
};
__device__ inline GRange px_g_range(const SPlan& P, int I) {
    int cost = 0;
    for (int j = 0; j < P.n; ++j) cost += (P.cnt[j] + 1) * I;
    const int beg = px_rp_at(P, I, int((long long)blockIdx.x * cost / gridDim.x));
    const int end = px_rp_at(P, I, int((long long)(blockIdx.x + 1) * cost / gridDim.x));
    return GRange{beg / I, beg % I, end - beg};
}

// A position in a ring of S slots, advanced one slot at a time (no division
// on the way: the loops that walk a ring run once per stage).
struct RingPos {
    int slot;
    uint32_t round;
    __device__ void next(int S) {
        if (++slot == S) {
            slot = 0;
            ++round;
        }
    }
};

// ------------------------------------------------------------- dot products
// Activations of token t in shared memory, chunk-interleaved: the 16-byte
// piece v of 32-element chunk c at piece index v * NC + c.

// One bf16 router row (natural layout, shared memory) against token x:
// four fp32 chains (even words' low and high halves, odd words' low and
// high halves), both operands bf16.
template <int MC>
__device__ __forceinline__ float px_router_dot(uint32_t wrow, uint32_t xrow, int NC, int lane) {
    float c0 = 0.0f, c1 = 0.0f, c2 = 0.0f, c3 = 0.0f;
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        if (c < NC) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 wu = lds128(wrow + 64u * c + 16u * v);
                const uint4 xu = lds128(xrow + 16u * (v * NC + c));
                c0 = fma_bf16<false, false>(wu.x, xu.x, c0);
                c1 = fma_bf16<true, true>(wu.x, xu.x, c1);
                c2 = fma_bf16<false, false>(wu.y, xu.y, c2);
                c3 = fma_bf16<true, true>(wu.y, xu.y, c3);
                c0 = fma_bf16<false, false>(wu.z, xu.z, c0);
                c1 = fma_bf16<true, true>(wu.z, xu.z, c1);
                c2 = fma_bf16<false, false>(wu.w, xu.w, c2);
                c3 = fma_bf16<true, true>(wu.w, xu.w, c3);
            }
        }
    }
    return warp_sum((c0 + c1) + (c2 + c3));
}

// Token x from shared memory: the lane's bf16 words of chunks lane and
// lane + 32.
template <int MC>
__device__ __forceinline__ void px_load_x(uint32_t xrow, int NC, int lane,
                                          uint32_t (&xb)[MC][16]) {
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        if (c < NC) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = lds128(xrow + 16u * (v * NC + c));
                xb[m][4 * v] = u.x;
                xb[m][4 * v + 1] = u.y;
                xb[m][4 * v + 2] = u.z;
                xb[m][4 * v + 3] = u.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) xb[m][j] = 0u;
        }
    }
}

// The fp32 sums of the same two chunks (the offset term of every group's
// dot product): taken once a layer, they serve every row.
template <int MC>
__device__ __forceinline__ float2 px_x_sums(uint32_t xrow, int NC, int lane) {
    float X[2] = {0.0f, 0.0f};
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        float sum = 0.0f;
        if (c < NC) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = lds128(xrow + 16u * (v * NC + c));
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) sum += bf16_lo(wv[i]) + bf16_hi(wv[i]);
            }
        }
        X[m] = sum;
    }
    return make_float2(X[0], X[1]);
}

// Rows r < nrows (<= NR) of length H (packed bytes at q + r * qs, fp16
// scales at s + r * ss, shared memory) against the token in xb / X, all at
// once: out[r] = the row's dot product, in every lane.
template <int MC, int NR>
__device__ __forceinline__ void px_rows_dot(uint32_t q, uint32_t s, uint32_t qs, uint32_t ss,
                                            int nrows, const uint32_t (&xb)[MC][16],
                                            const float (&X)[MC], int NC, int lane,
                                            float (&out)[NR]) {
    float acc[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r] = 0.0f;
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        if (c < NC) {
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r < nrows) {
                    const uint4 w = lds128(q + uint32_t(r) * qs + 16u * c);
                    const float sc = f16_to_f32(lds_u16(s + uint32_t(r) * ss + 2u * c));
                    acc[r] += group_dot128(dot_chunk_bf16(w, xb[m]), X[m], sc);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) out[r] = warp_sum(acc[r]);
}

// silu(gate) * up of one gate/up row pair (packed bytes at q, the up row at
// q + H/2; fp16 scales at s, the up row's at s + H/16; shared memory) for
// the token whose activations are at xrow, their chunk sums xs.  Out of line: phase R (the
// shared expert) and phase G (the routed experts) run the same instructions,
// so the second finds them in the instruction cache.
template <int MC>
__device__ __noinline__ float px_pair_silu(uint32_t q, uint32_t s, uint32_t xrow, float2 xs,
                                           int NC, int lane) {
    uint32_t xb[MC][16];
    px_load_x<MC>(xrow, NC, lane, xb);
    float X[MC];
    X[0] = xs.x;
    if constexpr (MC > 1) X[1] = xs.y;
    float gu[2];
    px_rows_dot<MC, 2>(q, s, uint32_t(NC) * 16u, uint32_t(NC) * 2u, 2, xb, X, NC, lane, gu);
    return silu_mul(gu[0], gu[1]);
}

// The routed and shared SwiGLU vectors of this layer (tagged words: TK rows
// of I at hr, T rows of Is at hs) into shared memory as fp32, every row
// chunk-interleaved (piece v of 32-element chunk c at piece v * (L/32) + c),
// by all consumer threads: a thread polls only its own pieces, all of them
// in flight, and again only those still missing.
__device__ void px_stage_h(const uint64_t* hr, const uint64_t* hs, uint32_t tag, int TK, int I,
                           int T, int Is, float* dst, int ctid, int nthr, uint32_t limit,
                           uint32_t* err) {
    const int pr = TK * (I / 4), ptot = pr + T * (Is / 4);     // pieces of four words
    constexpr int PB = 1;        // pieces a thread per batch (more cost registers: spills)
    for (int p0 = ctid; p0 < ptot; p0 += nthr * PB) {
        uint32_t todo = 0;
#pragma unroll
        for (int k = 0; k < PB; ++k)
            if (p0 + k * nthr < ptot) todo |= 1u << k;
        for (uint32_t it = 0; it < limit && todo != 0u; ++it) {
            uint64_t w[PB][4];
#pragma unroll
            for (int k = 0; k < PB; ++k) {
                if (todo & (1u << k)) {
                    const int p = p0 + k * nthr;
                    const uint64_t* src = p < pr ? hr + size_t(p) * 4 : hs + size_t(p - pr) * 4;
                    ll_ld2(src, w[k][0], w[k][1]);
                    ll_ld2(src + 2, w[k][2], w[k][3]);
                }
            }
#pragma unroll
            for (int k = 0; k < PB; ++k) {
                if ((todo & (1u << k)) && ll_has(w[k][0], tag) && ll_has(w[k][1], tag) &&
                    ll_has(w[k][2], tag) && ll_has(w[k][3], tag)) {
                    const int p = p0 + k * nthr;
                    const bool sh = p >= pr;
                    const int L = sh ? Is : I, q = sh ? p - pr : p;
                    const int row = q / (L / 4), e0 = (q % (L / 4)) * 4;
                    float* rowp = dst + (sh ? size_t(TK) * I + size_t(row) * Is : size_t(row) * I);
                    const int piece = ((e0 & 31) >> 2) * (L >> 5) + (e0 >> 5);
                    *reinterpret_cast<float4*>(rowp + 4 * piece) =
                        make_float4(ll_val(w[k][0]), ll_val(w[k][1]), ll_val(w[k][2]),
                                    ll_val(w[k][3]));
                    todo &= ~(1u << k);
                }
            }
            if (todo != 0u) {
                if ((it & 255u) == 255u && ld_relaxed_u32(err) == uint32_t(STRATA_ETIMEOUT)) break;
                px_backoff();
            }
        }
        if (todo != 0u) latch_timeout(err, 81, p0, tag, 0);
    }
}

// Down rows [r0, r1) of this CTA's rows of one unit (length L, packed bytes
// at sq, scales at ss, shared memory) for each slot s0 .. s0+scount-1 whose
// h row (fp32, chunk-interleaved, shared memory) is at hb + s * L * 4 bytes:
// s_y[(ybase + s) * R + row].  Lane (rs, c) holds chunk c of rows r0 + rs,
// r0 + rs + RPW, ... (RPW = 32 / chunks per row).
__device__ void px_down_unit(uint32_t sq, uint32_t ss, int L, int r0, int r1, int lane,
                             uint32_t hb, int s0, int scount, const int* tok, float* s_y,
                             int ybase, int R) {
    const int NCd = L >> 5, RPW = 32 / NCd;
    const int c = lane & (NCd - 1), rs = lane / NCd;
    const int nrow = r1 - r0;
    const int nr = (nrow > rs) ? (nrow - rs + RPW - 1) / RPW : 0;
    const int npass = (nrow + RPW - 1) / RPW;     // uniform over the warp
    const uint32_t qrow = uint32_t(L) >> 1, srow = uint32_t(L) >> 4;
    for (int si = 0; si < scount; ++si) {
        const int s = s0 + si;
        if (tok != nullptr && tok[s] < 0) continue;
        const uint32_t hrow = hb + uint32_t(s) * uint32_t(L) * 4u;
        uint64_t x2[16];
        float X = 0.0f;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = lds_f4(hrow + 16u * uint32_t(v * NCd + c));
            x2[2 * v] = pk(f.x, f.y);
            x2[2 * v + 1] = pk(f.z, f.w);
            X += (f.x + f.y) + (f.z + f.w);
        }
        // two rows of the lane a pass (npass is uniform over the warp)
#pragma unroll 1
        for (int m = 0; m < npass; m += 2) {
            float part[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int mm = m + k;
                part[k] = 0.0f;
                if (mm < nr) {
                    const uint32_t row = uint32_t(r0 + rs + mm * RPW);
                    const uint4 q = lds128(sq + row * qrow + 16u * c);
                    const float sc = f16_to_f32(lds_u16(ss + row * srow + 2u * c));
                    part[k] = group_dot(dot_chunk(q, x2), X, sc);
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int mm = m + k;
                if (mm < npass) {
                    const float v = group_sum(part[k], NCd);
                    if (c == 0 && mm < nr) s_y[size_t(ybase + s) * R + r0 + rs + mm * RPW] = v;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ kernel
// RESID: a residual stack (RMSNorm before each layer, the output added to
// the residual) or one layer on x_in; a kernel of each, so that one-layer
// calls carry no registers for the RMSNorm.
template <int MC, bool RESID>
__global__ void __launch_bounds__(kPxThreads, 1) k_persist(const __grid_constant__ PxArgs a) {
    extern __shared__ __align__(128) uint8_t px[];
    __shared__ SPlan P;
    __shared__ int s_ids[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_w[kDecodeMaxTokens * kMaxTopK];
    __shared__ int s_inv[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_sig[kDecodeMaxTokens];
    __shared__ float s_res[kPersistMaxTokens * 16];     // this CTA's rows of the residual
    __shared__ float s_den[kPersistMaxTokens];          // the RMSNorm denominators
    __shared__ __align__(8) uint64_t r_full, r_empty, plan_full, plan_free;
    __shared__ __align__(8) uint64_t sd_full[2], sd_empty[2];
    __shared__ __align__(8) uint64_t g_full[kPxGuMaxStages], g_empty[kPxGuMaxStages];
    __shared__ __align__(8) uint64_t d_full[kPxDnMaxStages], d_empty[kPxDnMaxStages];

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int T = a.T, H = a.H, E = a.E, K = a.K, I = a.I, Is = a.Is, TK = T * K;
    const int G = int(gridDim.x), b = int(blockIdx.x);
    const int NC = H >> 5;
    const int R = a.R, o0 = b * R;
    const int nrow = max(0, min(R, H - o0));
    // down products: a task is one pass of a warp over one unit (RPW rows,
    // 32 / chunks-per-row); every unit has max(1, passes) tasks, each
    // arriving once on the unit's empty barrier
    const int rpw_r = 32 / (I >> 5), rpw_s = 32 / (Is >> 5);
    const int np_r = max(1, (nrow + rpw_r - 1) / rpw_r), np_s = max(1, (nrow + rpw_s - 1) / rpw_s);
    const int Sg = a.gu_stages, Sd = a.dn_stages;
    const int nR = a.forced_ids ? 1 : E + 1;
    const uint32_t base = smem_u32(px);
    const uint32_t sx = base + a.off_x, sr = base + a.off_r, sg = base + a.off_g;
    const uint32_t sd0 = base + a.off_d;
    float* s_y = reinterpret_cast<float*>(px + a.off_y);
    uint32_t* err = a.err;

    pdl_launch();
    if (tid == 0) {
        mbar_init(&r_full, 1);
        mbar_init(&r_empty, 1);
        mbar_init(&plan_full, 1);
        mbar_init(&plan_free, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sd_full[i], 1);
            mbar_init(&sd_empty[i], np_s);            // one arrival a task
        }
        for (int i = 0; i < Sg; ++i) {
            mbar_init(&g_full[i], 1);
            mbar_init(&g_empty[i], 1);
        }
        for (int i = 0; i < Sd; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], np_r);             // one arrival a task
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (tid == 32) px_trace(0, a.n_layers, 0);

    const RShare rsh = px_r_share(b, G, nR, Is, H);

    // ================================================================ producer
    // (lane 0 the routing-independent rows; every lane its share of the
    // gate/up stages and down units, so the copies are requested in parallel)
    if (wid == 0) {
        // routing-independent rows of layer l: router + shared gate/up (R
        // buffer), shared down rows (SD buffer l & 1)
        auto issue_r = [&](int l) {
            const PxLayer& Lr = a.L[l];
            const uint32_t rb = uint32_t(rsh.nr) * 2u * H, qb = uint32_t(rsh.np) * H,
                           sb = uint32_t(rsh.np) * (H / 8);
            mbar_expect_tx(&r_full, rb + qb + sb);
            uint8_t* dst = px + a.off_r;
            const int r0 = a.forced_ids ? E : rsh.r0;
            if (rb) bulk_g2s(dst, Lr.router + size_t(r0) * H, rb, &r_full);
            if (qb) {
                bulk_g2s(dst + rb, Lr.sh_gu_q + size_t(2) * rsh.p0 * (H / 2), qb, &r_full);
                bulk_g2s(dst + rb + qb, Lr.sh_gu_s + size_t(2) * rsh.p0 * (H / 32), sb, &r_full);
            }
        };
        auto issue_sd = [&](int l) {
            const PxLayer& Lr = a.L[l];
            const int buf = l & 1;
            if (l >= 2 && !px_wait(&sd_empty[buf], ((l >> 1) - 1) & 1, err))
                latch_timeout(err, 64, buf, l, 0);
            const uint32_t qb = uint32_t(nrow) * (Is / 2), sb = uint32_t(nrow) * (Is / 16);
            mbar_expect_tx(&sd_full[buf], qb + sb);
            uint8_t* dst = px + a.off_sd + size_t(buf) * a.sd_bytes;
            if (qb) {
                bulk_g2s(dst, Lr.sh_dn_q + size_t(o0) * (Is / 2), qb, &sd_full[buf]);
                bulk_g2s(dst + a.sd_q, Lr.sh_dn_s + size_t(o0) * (Is / 32), sb, &sd_full[buf]);
            }
        };
        if (lane == 0) {
            issue_r(0);
            issue_sd(0);
        }
        RingPos gpos{0, 0}, dpos{0, 0};
        for (int l = 0; l < a.n_layers; ++l) {
            const PxLayer& Lr = a.L[l];
            if (!px_wait(&plan_full, l & 1, err)) latch_timeout(err, 60, 0, l, 0);
            px_fence_proxy_async();
            if (lane == 0) px_trace(l, a.n_layers, 11);
            // gate/up stages of this CTA's share, then its down rows of every
            // touched expert.  The first S of them (S the ring's slots) reuse
            // slots last filled in an earlier layer, whose consumers are done
            // (they finished before this layer's plan): lane k requests copy k
            // at once, its wait on the slot returning at once.  A copy past
            // the ring reuses a slot of this layer: lane 0 requests those, in
            // order, while the other lanes wait at the warp barrier -- so no
            // lane ever waits while another still has a copy to request that
            // the wait depends on.
            const GRange gr = px_g_range(P, I);
            const uint32_t dqb = uint32_t(nrow) * (I / 2), dsb = uint32_t(nrow) * (I / 16);
            auto issue_g = [&](int slot, int j, int i0, int nb) {
                uint8_t* dst = px + a.off_g + size_t(slot) * a.g_stage;
                const size_t row = size_t(P.e[j]) * 2 * I + size_t(2) * i0;
                const uint32_t qb = uint32_t(nb) * H, sb = uint32_t(nb) * (H / 8);
                mbar_expect_tx(&g_full[slot], qb + sb);
                bulk_g2s(dst, Lr.gu_q + row * (H / 2), qb, &g_full[slot]);
                bulk_g2s(dst + a.g_q, Lr.gu_s + row * (H / 32), sb, &g_full[slot]);
            };
            auto issue_d = [&](int slot, int j) {
                mbar_expect_tx(&d_full[slot], dqb + dsb);
                if (dqb) {
                    uint8_t* dst = px + a.off_d + size_t(slot) * a.d_stage;
                    const size_t row = size_t(P.e[j]) * H + o0;
                    bulk_g2s(dst, Lr.dn_q + row * (I / 2), dqb, &d_full[slot]);
                    bulk_g2s(dst + a.d_q, Lr.dn_s + row * (I / 32), dsb, &d_full[slot]);
                }
            };
            int nst = 0;                                 // this layer's stages
            for (int j = gr.j, i0 = gr.i0, left = gr.n; left > 0; ++j, i0 = 0) {
                const int seg = min(I - i0, left);
                nst += (seg + kPxRowPairs - 1) / kPxRowPairs;
                left -= seg;
            }
            const int ng0 = min(nst, Sg);
            for (int k = lane; k < ng0; k += 32) {
                const int sl = gpos.slot + k;               // < 2 Sg
                const int slot = sl < Sg ? sl : sl - Sg;
                const uint32_t round = gpos.round + (sl < Sg ? 0u : 1u);
                if (round > 0 && !px_wait(&g_empty[slot], (round - 1) & 1, err))
                    latch_timeout(err, 61, slot, round, l);
                // stage k: walk the range's expert segments to it
                int j = gr.j, i0 = gr.i0, left = gr.n, kk = k;
                for (;;) {
                    const int seg = min(I - i0, left);
                    const int ns = (seg + kPxRowPairs - 1) / kPxRowPairs;
                    if (kk < ns) {
                        i0 += kk * kPxRowPairs;
                        issue_g(slot, j, i0, min(kPxRowPairs, seg - kk * kPxRowPairs));
                        break;
                    }
                    kk -= ns;
                    left -= seg;
                    ++j;
                    i0 = 0;
                }
            }
            __syncwarp();
            if (nst > ng0) {
                if (lane == 0) {
                    RingPos pos = gpos;
                    int k = 0;
                    for (int j = gr.j, i0 = gr.i0, left = gr.n; left > 0; pos.next(Sg), ++k) {
                        const int nb = min(kPxRowPairs, min(I - i0, left));
                        if (k >= ng0) {
                            if (!px_wait(&g_empty[pos.slot], (pos.round - 1) & 1, err))
                                latch_timeout(err, 61, pos.slot, pos.round, l);
                            issue_g(pos.slot, j, i0, nb);
                        }
                        i0 += nb;
                        left -= nb;
                        if (i0 == I) {
                            ++j;
                            i0 = 0;
                        }
                    }
                }
                __syncwarp();
            }
            for (int k = 0; k < nst; ++k) gpos.next(Sg);
            if (lane == 0) px_trace(l, a.n_layers, 12);
            // the down units: the same split
            const int nd0 = min(P.n, Sd);
            for (int j = lane; j < nd0; j += 32) {
                const int sl = dpos.slot + j;
                const int slot = sl < Sd ? sl : sl - Sd;
                const uint32_t round = dpos.round + (sl < Sd ? 0u : 1u);
                if (round > 0 && !px_wait(&d_empty[slot], (round - 1) & 1, err))
                    latch_timeout(err, 62, slot, round, l);
                issue_d(slot, j);
            }
            __syncwarp();
            if (P.n > nd0) {
                if (lane == 0) {
                    RingPos pos = dpos;
                    for (int j = 0; j < P.n; ++j, pos.next(Sd)) {
                        if (j < nd0) continue;
                        if (!px_wait(&d_empty[pos.slot], (pos.round - 1) & 1, err))
                            latch_timeout(err, 62, pos.slot, pos.round, l);
                        issue_d(pos.slot, j);
                    }
                }
                __syncwarp();
            }
            for (int j = 0; j < P.n; ++j) dpos.next(Sd);
            if (lane == 0) px_trace(l, a.n_layers, 13);
            if (lane == 0) {
                mbar_arrive(&plan_free);          // P no longer read here
                // the next layer's routing-independent rows
                if (l + 1 < a.n_layers) {
                    if (!px_wait(&r_empty, l & 1, err)) latch_timeout(err, 63, 0, l, 0);
                    issue_r(l + 1);
                    issue_sd(l + 1);
                }
            }
        }
        // let every copy this CTA requested land before it exits: the last
        // round of every slot used.  These waits do not give up when another
        // wait ran out: shared memory must not be left with copies in flight.
        __syncwarp();
        if (lane != 0) return;
        for (int i = 0; i < Sg; ++i) {
            const uint32_t r = i < gpos.slot ? gpos.round : gpos.round - 1;
            if (i < gpos.slot || gpos.round > 0) mbar_wait(&g_full[i], r & 1);
        }
        for (int i = 0; i < Sd; ++i) {
            const uint32_t r = i < dpos.slot ? dpos.round : dpos.round - 1;
            if (i < dpos.slot || dpos.round > 0) mbar_wait(&d_full[i], r & 1);
        }
        const int nl = a.n_layers;
        mbar_wait(&r_full, (nl - 1) & 1);
        mbar_wait(&sd_full[(nl - 1) & 1], ((nl - 1) >> 1) & 1);
        if (nl >= 2) mbar_wait(&sd_full[nl & 1], ((nl - 2) >> 1) & 1);
        return;
    }

    // =============================================================== consumers
    const int cw = wid - 1, ctid = tid - 32;
    constexpr int NT = kPxConsumers * 32;
    const uint32_t lim = a.grid_wait_limit;
    pdl_wait();
    if (ctid == 0) px_trace(0, a.n_layers, 1);
    // the workspace's exchange count: this launch's tags follow it
    const uint32_t tag0 = ld_relaxed_u32(a.flags + b);
    auto tag = [&](int l, int ex) { return tag0 + uint32_t(kPxExchanges * l + ex) + 1u; };
    RingPos gpos{0, 0}, dpos{0, 0};
    for (int l = 0; l < a.n_layers; ++l) {
        const PxLayer& Lr = a.L[l];
        const bool last = l + 1 == a.n_layers;
        // ---- the layer input x (bf16) into shared memory
        if constexpr (RESID) {
            // RMSNorm of the residual: the caller's (plain) before the first
            // layer, the previous layer's tagged words after it.  Every
            // consumer thread gathers eight elements at once (one round trip
            // for the whole vector), parked as fp32 at the start of the
            // gate/up ring (idle between the layer's down products and its
            // next gate/up); then warp t reduces token t in the lane order
            // of the one-warp norm.
            float* raw = reinterpret_cast<float*>(px + a.off_g);
            const uint32_t tg = tag(l - 1, 2);
            for (int g = ctid; g < T * (H / 8); g += NT) {
                const int t = g / (H / 8), h = (g - t * (H / 8)) * 8;
                float4 v0, v1;
                if (l == 0) {
                    v0 = ldcg_f4(a.resid + size_t(t) * H + h);
                    v1 = ldcg_f4(a.resid + size_t(t) * H + h + 4);
                } else {
                    const uint64_t* lt = a.ll_resid + size_t(t) * H + h;
                    bool ok = false;
                    uint64_t w[8];
                    for (uint32_t it = 0; it < lim && !ok; ++it) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) ll_ld2(lt + 2 * i, w[2 * i], w[2 * i + 1]);
                        ok = true;
#pragma unroll
                        for (int i = 0; i < 8; ++i) ok &= ll_has(w[i], tg);
                        if (!ok && (it & 255u) == 255u &&
                            ld_relaxed_u32(err) == uint32_t(STRATA_ETIMEOUT))
                            break;
                        if (!ok) px_backoff();
                    }
                    if (!ok) latch_timeout(err, 83, t, l, h);
                    v0 = make_float4(ll_val(w[0]), ll_val(w[1]), ll_val(w[2]), ll_val(w[3]));
                    v1 = make_float4(ll_val(w[4]), ll_val(w[5]), ll_val(w[6]), ll_val(w[7]));
                }
                *reinterpret_cast<float4*>(raw + size_t(t) * H + h) = v0;
                *reinterpret_cast<float4*>(raw + size_t(t) * H + h + 4) = v1;
            }
            px_cbar();
            // this CTA's rows of it, for the residual add after the combine
            for (int i = ctid; i < T * nrow; i += NT) {
                const int t = i / nrow, r = i - t * nrow;
                s_res[t * 16 + r] = raw[size_t(t) * H + o0 + r];
            }
            for (int t = cw; t < T; t += kPxConsumers) {
                const float* rw = raw + size_t(t) * H;
                float ss = 0.0f;
#pragma unroll 1
                for (int h0 = lane * 4; h0 < H; h0 += 128 * 4) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (h0 + 128 * i < H) {
                            const float4 v = *reinterpret_cast<const float4*>(rw + h0 + 128 * i);
                            ss += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
                        }
                    }
                }
                ss = warp_sum(ss);
                if (lane == 0) s_den[t] = sqrtf(ss / float(H) + a.eps);
            }
            px_cbar();
            // the normalised token rows into shared memory (bf16, chunk-interleaved)
            for (int i = ctid; i < T * (H / 4); i += NT) {
                const int t = i / (H / 4), h = (i - t * (H / 4)) * 4;
                const float denom = s_den[t];
                const float4 v = *reinterpret_cast<const float4*>(raw + size_t(t) * H + h);
                const uint32_t p0 = uint32_t(f32_to_bf16(v.x / denom)) |
                                    (uint32_t(f32_to_bf16(v.y / denom)) << 16);
                const uint32_t p1 = uint32_t(f32_to_bf16(v.z / denom)) |
                                    (uint32_t(f32_to_bf16(v.w / denom)) << 16);
                const int c = h >> 5, v8 = (h & 31) >> 3;
                uint8_t* xt = px + a.off_x + size_t(t) * H * 2;
                *reinterpret_cast<uint2*>(xt + 16 * (v8 * NC + c) + 2 * (h & 7)) =
                    make_uint2(p0, p1);
                if (a.x_out != nullptr && b == 0 && last)
                    *reinterpret_cast<uint2*>(a.x_out + size_t(t) * H + h) = make_uint2(p0, p1);
            }
        } else {
            uint4* xs = reinterpret_cast<uint4*>(px + a.off_x);
            for (int i = ctid; i < T * 4 * NC; i += NT) {
                const int t = i / (4 * NC), r = i - t * 4 * NC, c = r >> 2, v = r & 3;
                xs[size_t(t) * 4 * NC + v * NC + c] =
                    __ldcg(reinterpret_cast<const uint4*>(a.x_in + size_t(t) * H) + 4 * c + v);
            }
        }
        px_cbar();
        // the token's chunk sums, for every gate/up row pair of the layer
        static_assert(kPersistMaxTokens == 1, "one token's chunk sums a layer");
        const float2 xsum = px_x_sums<MC>(sx, NC, lane);
        if (ctid == 0) px_trace(l, a.n_layers, 2);

        // ---- R: router rows and shared gate/up row pairs of this CTA
        if (!px_wait(&r_full, l & 1, err)) latch_timeout(err, 71, 0, l, 0);
        {
            const uint32_t tg_l = tag(l, 0), tg_s = tag(l, 1);   // logits; SwiGLU vectors
            const uint32_t rq = sr + uint32_t(rsh.nr) * 2u * H;
            const uint32_t rs_ = rq + uint32_t(rsh.np) * H;
            for (int u = cw; u < rsh.nr + rsh.np; u += kPxConsumers) {
                if (u < rsh.nr) {
                    const int e = a.forced_ids ? E : rsh.r0 + u;
                    const float bias = (e < E && Lr.bias != nullptr) ? __ldg(Lr.bias + e) : 0.0f;
                    const uint32_t wrow = sr + uint32_t(u) * 2u * H;
                    for (int t = 0; t < T; ++t) {
                        const float v = px_router_dot<MC>(wrow, sx + uint32_t(t) * H * 2, NC, lane);
                        if (lane == 0) ll_put(a.ll_logits + size_t(t) * (E + 1) + e, v + bias, tg_l);
                    }
                } else {
                    const int pl = u - rsh.nr, p = rsh.p0 + pl;
                    const uint32_t qg = rq + uint32_t(2 * pl) * (H / 2);
                    const uint32_t sgs = rs_ + uint32_t(2 * pl) * (H / 16);
                    for (int t = 0; t < T; ++t) {
                        const float hv = px_pair_silu<MC>(qg, sgs, sx + uint32_t(t) * H * 2, xsum,
                                                          NC, lane);
                        if (lane == 0) ll_put(a.ll_hs + size_t(t) * Is + p, hv, tg_s);
                    }
                }
            }
        }
        px_cbar();
        if (ctid == 0) {
            px_trace(l, a.n_layers, 3);
            mbar_arrive(&r_empty);
        }

        // ---- S: selection and bucketing (the same in every CTA)
        if (l > 0 && ctid == 0 && !px_wait(&plan_free, (l - 1) & 1, err))
            latch_timeout(err, 73, 0, l, 0);
        {
            const uint32_t tg_l = tag(l, 0);
            uint32_t* keys = reinterpret_cast<uint32_t*>(px + a.off_g);
            for (int t = cw; t < T; t += kPxConsumers) {
                const uint64_t* lg = a.ll_logits + size_t(t) * (E + 1);
                uint32_t* Lk = keys + size_t(cw) * (E + 16);
                // every logit of the token (and the gate logit, entry E),
                // polled until all carry this layer's tag
                float gl = 0.0f;
                bool ok = false;
                // forced routing computes the gate row E only
                const bool fr = a.forced_ids != nullptr;
                for (uint32_t it = 0; it < lim && !ok; ++it) {
                    bool mine = true;
#pragma unroll 1
                    for (int e0 = fr ? E - (E & 31) : 0; e0 <= E; e0 += 32 * 9) {
                        uint64_t w[9];
#pragma unroll
                        for (int j = 0; j < 9; ++j) {
                            const int e = e0 + lane + 32 * j;
                            w[j] = (e <= E && (!fr || e == E)) ? ll_ld(lg + e)
                                                                : uint64_t(tg_l) << 32;
                        }
#pragma unroll
                        for (int j = 0; j < 9; ++j) {
                            const int e = e0 + lane + 32 * j;
                            mine &= ll_has(w[j], tg_l);
                            if (e < E && !fr)
                                Lk[e] = logit_key(ll_val(w[j]));
                            else if (e == E)
                                gl = ll_val(w[j]);
                        }
                    }
                    ok = __all_sync(0xffffffffu, mine);
                    if (!ok && (it & 255u) == 255u &&
                        ld_relaxed_u32(err) == uint32_t(STRATA_ETIMEOUT))
                        break;
                    if (!ok) px_backoff();
                }
                if (!ok && lane == 0) latch_timeout(err, 80, t, tg_l, 0);
                if (t == 0 && lane == 0) px_trace(l, a.n_layers, 4);
                gl = __shfl_sync(0xffffffffu, gl, E & 31);
                if (a.forced_ids != nullptr) {
                    const int32_t* fi = a.forced_ids + size_t(l) * TK + size_t(t) * K;
                    const float* fw = a.forced_w + size_t(l) * TK + size_t(t) * K;
                    for (int k = lane; k < K; k += 32) {
                        const int id = __ldg(fi + k);
                        if (id < 0 || id >= E) latch(err, STRATA_EBADROUTE);
                        s_ids[t * K + k] = id;
                        s_w[t * K + k] = __ldg(fw + k);
                    }
                } else {
                    select_topk_keys(E, K, Lk, reinterpret_cast<float*>(Lk + E), s_ids + t * K,
                                     s_w + t * K, lane);
                }
                if (lane == 0) s_sig[t] = 1.0f / (1.0f + expf(-gl));
                if (t == 0 && lane == 0) px_trace(l, a.n_layers, 5);
            }
        }
        px_cbar();
        {
            int* s_cnt = reinterpret_cast<int*>(px + a.off_g);
            int* s_off = s_cnt + E;
            int* s_wsum = s_off + E + 1;
            const BucketOut none{nullptr, nullptr, nullptr, nullptr, nullptr};
            // one token whose ids ascend (the selection's order): slot k is
            // pick k, the plan is the ids themselves
            bool trivial = false;
            if (T == 1) {
                const int id = lane < K ? s_ids[lane] : 0x7fffffff;
                const int prev = __shfl_up_sync(0xffffffffu, id, 1);
                trivial = __all_sync(0xffffffffu, lane >= K || ((lane == 0 || prev < id) && id >= 0 &&
                                                                id < E));
            }
            if (trivial) {
                if (cw == 0) {
                    if (lane < K) {
                        P.e[lane] = s_ids[lane];
                        P.off[lane] = lane;
                        P.cnt[lane] = 1;
                        P.tok[lane] = 0;
                        s_inv[lane] = lane;
                    }
                    if (lane == 0) P.n = K;
                }
            } else {
                bucket_cta(s_ids, T, K, E, s_cnt, s_off, s_wsum, P, s_inv, none, ctid, NT,
                           PxSync{});
            }
        }
        px_fence_proxy_async();
        px_cbar();
        if (ctid == 0) {
            mbar_arrive(&plan_full);
            px_trace(l, a.n_layers, 6);
        }

        // ---- G: gate/up + SwiGLU, one warp a stage of this CTA's row pairs
        {
            const uint32_t tg_h = tag(l, 1);
            const GRange gr = px_g_range(P, I);
            for (int j = gr.j, i0 = gr.i0, left = gr.n; left > 0; gpos.next(Sg)) {
                const int nb = min(kPxRowPairs, min(I - i0, left));
                const int slot = gpos.slot;
                const uint32_t round = gpos.round;
                const int ji = j, ii0 = i0;
                i0 += nb;
                left -= nb;
                if (i0 == I) {
                    ++j;
                    i0 = 0;
                }
                if (slot % kPxConsumers != cw) continue;       // another warp's stage
                if (!px_wait(&g_full[slot], round & 1, err)) latch_timeout(err, 74, slot, round, l);
                const uint32_t sq = sg + uint32_t(slot) * a.g_stage, ssc = sq + a.g_q;
                const int s0 = P.off[ji], scount = P.cnt[ji];
                for (int si = 0; si < scount; ++si) {
                    const int s = s0 + si, t = P.tok[s];
                    if (t < 0 || t >= T) continue;
#pragma unroll 1
                    for (int p = 0; p < nb; ++p) {
                        const float hv = px_pair_silu<MC>(sq + uint32_t(p) * H,
                                                          ssc + uint32_t(p) * (H / 8),
                                                          sx + uint32_t(t) * H * 2, xsum, NC, lane);
                        if (lane == 0) ll_put(a.ll_h + size_t(s) * I + ii0 + p, hv, tg_h);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&g_empty[slot]);
            }
        }

        // ---- D: down products of this CTA's output rows, then the combine
        {
            const uint32_t tg_h = tag(l, 1), tg_r = tag(l, 2);
            const int n = P.n;
            for (int i = ctid; i < (TK + T) * R; i += NT) s_y[i] = 0.0f;
            // every warp's gate/up stages are computed: the ring holds h now
            px_cbar();
            if (ctid == 0) px_trace(l, a.n_layers, 7);
            float* hsm = reinterpret_cast<float*>(px + a.off_g);
            px_stage_h(a.ll_h, a.ll_hs, tg_h, TK, I, T, Is, hsm, ctid, NT, lim, err);
            px_cbar();
            if (ctid == 0) px_trace(l, a.n_layers, 8);
            const uint32_t hb = sg;
            // tasks: first the shared unit's np_s passes, then np_r passes of
            // each routed unit j (in the ring's order: unit j in the slot j
            // places after this layer's first).  Warp w takes the contiguous
            // run [w * ntask / 15, (w + 1) * ntask / 15), at most a few units,
            // each as one call (its h loaded once, two rows a lane in flight);
            // it arrives on a unit's empty barrier once per task it took.  A
            // task's wait only depends on tasks of lower index (the unit's
            // earlier round in the same slot), and every warp takes its run in
            // increasing order, so the lowest unfinished task can always run.
            const int ntask = np_s + n * np_r;
            const int k1 = (cw + 1) * ntask / kPxConsumers;
            RingPos up = dpos;                 // the slot of routed unit uj
            int uj = 0;
            for (int k = cw * ntask / kPxConsumers; k < k1;) {
                if (k < np_s) {
                    const int kend = min(k1, np_s);
                    const int buf = l & 1;
                    if (!px_wait(&sd_full[buf], (l >> 1) & 1, err))
                        latch_timeout(err, 77, buf, l, 0);
                    const uint32_t dq = base + a.off_sd + uint32_t(buf) * a.sd_bytes;
                    const int r0 = k * rpw_s, r1 = min(kend * rpw_s, nrow);
                    if (r1 > r0)
                        px_down_unit(dq, dq + a.sd_q, Is, r0, r1, lane,
                                     hb + uint32_t(TK) * uint32_t(I) * 4u, 0, T, nullptr, s_y, TK,
                                     R);
                    __syncwarp();
                    if (lane == 0) mbar_arrive_n(&sd_empty[buf], uint32_t(kend - k));
                    k = kend;
                } else {
                    const int j = (k - np_s) / np_r, p0 = (k - np_s) - j * np_r;
                    const int kend = min(k1, np_s + (j + 1) * np_r);
                    const int p1 = kend - np_s - j * np_r;
                    for (; uj < j; ++uj) up.next(Sd);
                    if (!px_wait(&d_full[up.slot], up.round & 1, err))
                        latch_timeout(err, 76, up.slot, up.round, l);
                    const uint32_t dq = sd0 + uint32_t(up.slot) * a.d_stage;
                    const int r0 = p0 * rpw_r, r1 = min(p1 * rpw_r, nrow);
                    if (r1 > r0)
                        px_down_unit(dq, dq + a.d_q, I, r0, r1, lane, hb, P.off[j], P.cnt[j],
                                     P.tok, s_y, 0, R);
                    __syncwarp();
                    if (lane == 0) mbar_arrive_n(&d_empty[up.slot], uint32_t(kend - k));
                    k = kend;
                }
            }
            for (int j = 0; j < n; ++j) dpos.next(Sd);
            px_cbar();
            if (ctid == 0) px_trace(l, a.n_layers, 9);
            const bool write_out = a.out != nullptr && (last || !RESID);
            for (int i = ctid; i < T * nrow; i += NT) {
                const int t = i / nrow, r = i - t * nrow, o = o0 + r;
                float acc = 0.0f;
                for (int k = 0; k < K; ++k) {
                    const int sl = s_inv[t * K + k];
                    if (sl < 0 || sl >= TK) continue;
                    acc += s_w[t * K + k] * s_y[size_t(sl) * R + r];
                }
                const float v = acc + s_sig[t] * s_y[size_t(TK + t) * R + r];
                const uint16_t ob = f32_to_bf16(v);
                if (write_out) a.out[size_t(t) * H + o] = ob;
                if constexpr (RESID) {
                    float* rp = a.resid + size_t(t) * H + o;
                    const float rn = s_res[t * 16 + r] + __uint_as_float(uint32_t(ob) << 16);
                    *rp = rn;
                    if (!last) ll_put(a.ll_resid + size_t(t) * H + o, rn, tg_r);
                }
            }
        }
        if (ctid == 0) px_trace(l, a.n_layers, 10);
        // the last layer's routing and bucketing, by the last CTA (the one
        // with the fewest output rows, done first), so that no CTA with a
        // full share of the down products ends later for it
        if (last && b == G - 1) {
            publish_bucket(TK, E, P, s_inv, BucketOut{a.counts, a.offsets, a.perm, a.inv, nullptr},
                           ctid, NT);
            for (int p = ctid; p < TK; p += NT) {
                a.ids[p] = s_ids[p];
                a.w[p] = s_w[p];
                if (a.ids_user) a.ids_user[p] = s_ids[p];
                if (a.w_user) a.w_user[p] = s_w[p];
            }
            for (int t = ctid; t < T; t += NT) {
                a.sig[t] = s_sig[t];
                if (a.sig_user) a.sig_user[t] = s_sig[t];
            }
        }
    }
    // this launch's exchanges are spent: the next launch's tags follow them
    if (ctid == 0) a.flags[b] = tag0 + uint32_t(kPxExchanges * a.n_layers);
}

// ------------------------------------------------------------------ launch
cudaError_t px_trace_copy(void* host, size_t bytes) {
#ifdef STRATA_PX_TRACE
    if (bytes > kPxTraceBytes) bytes = kPxTraceBytes;
    return cudaMemcpyFromSymbol(host, g_px_trace, bytes);
#else
    (void)host;
    (void)bytes;
    return cudaErrorNotSupported;
#endif
}

namespace {

size_t align128(size_t x) { return (x + 127) & ~size_t(127); }

using PxFn = void (*)(PxArgs);

PxFn px_kernel(int MC, bool resid) {
    if (resid) return MC == 1 ? k_persist<1, true> : k_persist<2, true>;
    return MC == 1 ? k_persist<1, false> : k_persist<2, false>;
}

}  // namespace

bool px_geometry(const strata_moe_dims& d, int T, bool forced, bool resid, int G, PxGeo* g) {
    const int H = d.hidden, E = d.n_experts, K = d.top_k, I = d.inter, Is = d.shared_inter;
    *g = PxGeo{};
    if (T < 1 || T > kPersistMaxTokens || T > kPersistTokensCap || H > 2048 || G < 1 ||
        G > kMaxGrid)
        return false;
    const int MC = H <= 1024 ? 1 : 2;
    const int q = 256 / (I < Is ? I : Is) > 1 ? 256 / (I < Is ? I : Is) : 1;
    int R = (H + G - 1) / G;
    R = (R + q - 1) / q * q;
    if (R > 16) return false;
    const int nR = forced ? 1 : E + 1;
    size_t rmax = 0;
    for (int b = 0; b < G; ++b) {
        const RShare s = px_r_share(b, G, nR, Is, H);
        const size_t bytes = size_t(s.nr) * 2 * H + size_t(s.np) * (H + H / 8);
        if (bytes > rmax) rmax = bytes;
    }
    g->MC = MC;
    g->R = R;
    g->sd_q = uint32_t(align128(size_t(R) * (Is / 2)));
    g->sd_bytes = uint32_t(align128(g->sd_q + size_t(R) * (Is / 16)));
    g->d_q = uint32_t(align128(size_t(R) * (I / 2)));
    g->d_stage = uint32_t(align128(g->d_q + size_t(R) * (I / 16)));
    g->g_q = uint32_t(size_t(kPxRowPairs) * H);
    g->g_stage = uint32_t(align128(g->g_q + size_t(kPxRowPairs) * (H / 8)));
    const size_t x_bytes = align128(size_t(T) * H * 2);
    const size_t r_bytes = align128(rmax > 0 ? rmax : 16);
    const size_t y_bytes = align128(size_t(T * K + T) * R * 4);
    // the gate/up ring: a multiple of the consumer warps (stage k is computed
    // by warp (k mod ring) mod warps, so each slot's rounds are one warp's);
    // between the layer's gate/up stages it holds the selection's and the
    // bucketing's scratch, the RMSNorm's residual and the SwiGLU vectors the
    // down products read.  The down ring: all of a small call's units (and
    // the next one) in flight, within 40 KB and what the gate/up ring leaves.
    const size_t scratch = size_t(kPxConsumers) * (E + 16) * 4 > size_t(2 * E + 33) * 4
                               ? size_t(kPxConsumers) * (E + 16) * 4
                               : size_t(2 * E + 33) * 4;
    const size_t budget = kPxSmemBudget;
    const size_t fixed = x_bytes + r_bytes + size_t(2) * g->sd_bytes + y_bytes;
    const size_t g_round = size_t(kPxConsumers) * g->g_stage;
    if (fixed + g_round + size_t(2) * g->d_stage > budget) return false;
    int Sg = int((budget - fixed - size_t(2) * g->d_stage) / g_round) * kPxConsumers;
    if (Sg > kPxGuMaxStages) Sg = kPxGuMaxStages / kPxConsumers * kPxConsumers;
    if (size_t(Sg) * g->g_stage < scratch) return false;
    if (resid && size_t(Sg) * g->g_stage < size_t(T) * H * 4) return false;
    // the down products read the SwiGLU vectors from the same place
    if (size_t(Sg) * g->g_stage < (size_t(T) * K * I + size_t(T) * Is) * 4) return false;
    const int units = T * K < E ? T * K : E;
    int Sd = units + 1;
    const size_t d_room = budget - fixed - size_t(Sg) * g->g_stage;
    const size_t d_cap = d_room < (size_t(40) << 10) ? d_room : (size_t(40) << 10);
    if (Sd > int(d_cap / g->d_stage)) Sd = int(d_cap / g->d_stage);
    if (Sd > kPxDnMaxStages) Sd = kPxDnMaxStages;
    if (Sd < 2) return false;
    // a layer's gate/up stages and down units fit their rings in one round:
    // a CTA's share of T K I row pairs (cost-balanced: every one of the
    // token's units weighs the same) is at most ceil(K I / G) + 1 pairs, cut
    // at most once at an expert boundary.  (Rings that wrap inside a layer
    // take code paths that a multi-token run saw fail; they stay closed.)
    const int pairs_max = (K * I + G - 1) / G + 1;
    if ((pairs_max + kPxRowPairs - 1) / kPxRowPairs + 1 > Sg || units > Sd) return false;
    g->dn_stages = Sd;
    g->gu_stages = Sg;
    size_t o = 0;
    g->off_x = uint32_t(o);
    o += x_bytes;
    g->off_r = uint32_t(o);
    o += r_bytes;
    g->off_sd = uint32_t(o);
    o += size_t(2) * g->sd_bytes;
    g->off_d = uint32_t(o);
    o += size_t(Sd) * g->d_stage;
    g->off_y = uint32_t(o);
    o += y_bytes;
    g->off_g = uint32_t(align128(o));
    size_t dyn = g->off_g + size_t(Sg) * g->g_stage;
    if (dyn < kPxSmemMin) dyn = kPxSmemMin;       // one CTA per SM
    g->dyn = uint32_t(dyn);
    return true;
}

cudaError_t launch_persistent(const PxArgs& a, const PxGeo& g, cudaStream_t s) {
    PxFn fn = px_kernel(g.MC, a.resid != nullptr);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(g.dyn));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(device_info().sms);
    cfg.blockDim = dim3(kPxThreads);
    cfg.dynamicSmemBytes = g.dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, a);
    if (e == cudaSuccess) prof_after_launch(s);
    return e;
}

}  // namespace strata
