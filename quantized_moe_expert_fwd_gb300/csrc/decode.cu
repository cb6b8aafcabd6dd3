// decode.cu -- the decode-size (T <= 32) kernels of the routed MoE FFN.
//
// Three launches make one layer (Strata, "Qwen3.6-35B-A3B: pictures, several
// requests at once and speed", section "Speed": router top-k and grouping in
// one launch, the router and the shared gate in one product, shared
// gate+up+SwiGLU in one launch, the MoE end in one launch; PolyStrata,
// "Models and backends", section "What was tuned": a call's experts go
// through one launch per stage, and one launch adds them up):
//
//   k_route_decode  router rows (E+1 of them: the last is the shared-expert
//                   gate) and the shared expert's gate/up rows, spread over
//                   every SM; the last CTA to finish selects the top-K of
//                   each token, computes the renormalised softmax weights and
//                   the sigmoid gate, and buckets the (token, k) pairs by
//                   expert.
//   k_gate_up       every touched expert's gate/up rows, each read once for
//                   all tokens routed to it, with SwiGLU in the epilogue.
//   k_down          for a block of output rows: every touched expert's down
//                   rows and the shared expert's, then the weighted combine
//                   (or, as separate calls, per-slot outputs / the combine of
//                   given per-slot outputs).
//
// Weights stream through 128-bit non-allocating loads, each 16-byte chunk
// being one scale group of 32 int4 weights; dequantisation is the byte
// placement of common.cuh (no conversion instructions) and packed f32x2 FMAs.
// Every sum has a fixed order: results do not depend on timing.

#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace strata {

// ---------------------------------------------------------------- experts
// The touched experts, ascending, with their slot ranges.  Every CTA of the
// expert kernels builds it from `offsets`, so those kernels accept a
// bucketing from any source.
struct ActiveList {
    int n;
    int e[kMaxExperts];
    int off[kMaxExperts];
    int cnt[kMaxExperts];
};

__device__ void build_active(ActiveList& A, const int32_t* offsets, int E, int TK,
                             uint32_t* err) {
    __shared__ int warp_base[32];
    __shared__ int running;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0) running = 0;
    __syncthreads();
    for (int base = 0; base < E; base += blockDim.x) {
        const int e = base + tid;
        int off = 0, cnt = 0;
        if (e < E) {
            off = __ldcg(offsets + e);
            const int end = __ldcg(offsets + e + 1);
            cnt = end - off;
            if (off < 0 || cnt < 0 || end > TK) {
                latch(err, STRATA_EBADROUTE);
                cnt = 0;
            }
        }
        const unsigned bal = __ballot_sync(0xffffffffu, cnt > 0);
        const int pre = __popc(bal & ((1u << lane) - 1u));
        if (lane == 0) warp_base[wid] = __popc(bal);
        __syncthreads();
        if (tid == 0) {
            int r = running;
            for (int w = 0; w < nw; ++w) {
                const int c = warp_base[w];
                warp_base[w] = r;
                r += c;
            }
            running = r;
        }
        __syncthreads();
        if (cnt > 0) {
            const int pos = warp_base[wid] + pre;
            A.e[pos] = e;
            A.off[pos] = off;
            A.cnt[pos] = cnt;
        }
        __syncthreads();
    }
    if (tid == 0) A.n = running;
    __syncthreads();
}

// Lane `lane` owns chunks c = lane + 32 m (m < MC) of a length-H row; a chunk
// is 32 elements.  Loads token row x (bf16) as fp32 pairs plus chunk sums.
template <int MC>
__device__ __forceinline__ void load_x(const uint16_t* xrow, int NC, int lane,
                                       uint64_t (&x2)[MC][16], float (&X)[MC]) {
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        float sum = 0.0f;
        if (c < NC) {
            const uint4* p = reinterpret_cast<const uint4*>(xrow + 32 * c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = ldg_keep(p + v);
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = bf16_lo(wv[i]), hi = bf16_hi(wv[i]);
                    x2[m][4 * v + i] = pk(lo, hi);
                    sum += lo + hi;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) x2[m][j] = 0ull;
        }
        X[m] = sum;
    }
}

// Gate/up of row pairs [i0, i0 + nb) of one expert for the tokens of slots
// [s0, s0 + scount): h[s][i] = silu(g_i) u_i.  perm == nullptr means slot s
// is token s (the shared expert).  One warp.
template <int MC, int RB>
__device__ void gu_batch(const uint8_t* qe, const uint16_t* se, int H, int i0, int nb,
                         const uint16_t* x, int s0, int scount, const int32_t* perm, int K,
                         int TK, float* h, int ldh, uint32_t* err, int lane) {
    const int NC = H >> 5;
    const size_t qrow = size_t(H) >> 1;
    const size_t srow = size_t(H) >> 5;
    uint4 qv[RB][2][MC];
    float sc[RB][2][MC];
#pragma unroll
    for (int p = 0; p < RB; ++p)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int m = 0; m < MC; ++m) {
                const int c = lane + 32 * m;
                const size_t row = size_t(2 * (i0 + p) + r);
                if (p < nb && c < NC) {
                    qv[p][r][m] = ldg_stream(qe + row * qrow + size_t(c) * 16);
                    sc[p][r][m] = f16_to_f32(ldg_u16(se + row * srow + c));
                } else {
                    qv[p][r][m] = make_uint4(0u, 0u, 0u, 0u);
                    sc[p][r][m] = 0.0f;
                }
            }
    for (int si = 0; si < scount; ++si) {
        const int s = s0 + si;
        int t = s;
        if (perm != nullptr) {
            const int pr = __ldcg(perm + s);
            if (pr < 0 || pr >= TK) {
                latch(err, STRATA_EBADROUTE);
                continue;
            }
            t = pr / K;
        }
        uint64_t x2[MC][16];
        float X[MC];
        load_x<MC>(x + size_t(t) * H, NC, lane, x2, X);
        float acc[RB][2];
#pragma unroll
        for (int p = 0; p < RB; ++p)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float a = 0.0f;
#pragma unroll
                for (int m = 0; m < MC; ++m)
                    if (lane + 32 * m < NC)
                        a += group_dot(dot_chunk(qv[p][r][m], x2[m]), X[m], sc[p][r][m]);
                acc[p][r] = warp_sum(a);
            }
        float g = 0.0f, u = 0.0f;
#pragma unroll
        for (int p = 0; p < RB; ++p)
            if (p == lane) {
                g = acc[p][0];
                u = acc[p][1];
            }
        if (lane < nb) h[size_t(s) * ldh + i0 + lane] = silu_mul(g, u);
    }
}

// ------------------------------------------------------------- k_gate_up
template <int MC, int RB>
__global__ void __launch_bounds__(256, 1) k_gate_up(GuLaunch a) {
    __shared__ ActiveList s_act;
    const int lane = threadIdx.x & 31;
    const int TK = a.T * a.K;
    if (a.shared) {
        if (threadIdx.x == 0) {
            s_act.n = 1;
            s_act.e[0] = 0;
            s_act.off[0] = 0;
            s_act.cnt[0] = a.T;
        }
        __syncthreads();
    } else {
        build_active(s_act, a.offsets, a.E, TK, a.err);
    }
    const long long RP = (long long)s_act.n * a.I;
    const int wpb = blockDim.x >> 5;
    const long long NW = (long long)gridDim.x * wpb;
    const long long gw = (long long)blockIdx.x * wpb + (threadIdx.x >> 5);
    const long long beg = gw * RP / NW, end = (gw + 1) * RP / NW;
    const size_t qexp = size_t(2) * a.I * (size_t(a.H) >> 1);
    const size_t sexp = size_t(2) * a.I * (size_t(a.H) >> 5);
    for (long long rp = beg; rp < end;) {
        const int j = int(rp / a.I), i0 = int(rp % a.I);
        const int nb = int(min((long long)RB, min((long long)(a.I - i0), end - rp)));
        const int e = s_act.e[j];
        gu_batch<MC, RB>(a.q + size_t(e) * qexp, a.sc + size_t(e) * sexp, a.H, i0, nb, a.x,
                         s_act.off[j], s_act.cnt[j], a.shared ? nullptr : a.perm, a.K, TK, a.h,
                         a.I, a.err, lane);
        rp += nb;
    }
}

// Stable counting sort of the T*K (token, k) pairs by expert, one CTA.
// ids: the pairs' expert ids in shared memory; out-of-range ids get no slot
// (inv = -1).  counts[e], offsets[0..E], perm[slot] = t*K + k with the slots
// of one expert in ascending t, inv[t*K + k] = slot.
__device__ void permute_block(const int32_t* s_ids, int T, int K, int E, int32_t* counts,
                              int32_t* offsets, int32_t* perm, int32_t* inv, int* s_cnt,
                              int* s_off, int* s_wsum) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, wpb = blockDim.x >> 5;
    const int TK = T * K;
    for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    for (int p = tid; p < TK; p += blockDim.x) {
        const int e = s_ids[p];
        if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    }
    __syncthreads();
    // exclusive scan of s_cnt: each thread one contiguous segment of experts
    const int seg = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, tid * seg), e1 = min(E, e0 + seg);
    int local = 0;
    for (int e = e0; e < e1; ++e) local += s_cnt[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[wid] = incl;
    __syncthreads();
    if (tid == 0) {
        int r = 0;
        for (int w = 0; w < wpb; ++w) {
            const int c = s_wsum[w];
            s_wsum[w] = r;
            r += c;
        }
        s_off[E] = r;
    }
    __syncthreads();
    int run = s_wsum[wid] + incl - local;
    for (int e = e0; e < e1; ++e) {
        s_off[e] = run;
        run += s_cnt[e];
    }
    __syncthreads();
    for (int p = tid; p < TK; p += blockDim.x) {
        const int e = s_ids[p];
        if (e < 0 || e >= E) inv[p] = -1;
    }
    for (int e = tid; e < E; e += blockDim.x) {
        const int c = s_cnt[e];
        counts[e] = c;
        offsets[e] = s_off[e];
        if (c == 0) continue;
        int slot = s_off[e];
        for (int p = 0; p < TK; ++p)
            if (s_ids[p] == e) {
                perm[slot] = p;
                inv[p] = slot;
                ++slot;
            }
    }
    if (tid == 0) offsets[E] = s_off[E];
}

// Standalone bucketing of up to kDecodeMaxTokens * kMaxTopK pairs.
__global__ void __launch_bounds__(256, 1) k_permute_small(const int32_t* ids, int T, int K, int E,
                                                          int32_t* counts, int32_t* offsets,
                                                          int32_t* perm, int32_t* inv,
                                                          uint32_t* err) {
    __shared__ int32_t s_ids[kDecodeMaxTokens * kMaxTopK];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_wsum[32];
    for (int p = threadIdx.x; p < T * K; p += blockDim.x) {
        const int e = __ldg(ids + p);
        if (e < 0 || e >= E) latch(err, STRATA_EBADROUTE);
        s_ids[p] = e;
    }
    __syncthreads();
    permute_block(s_ids, T, K, E, counts, offsets, perm, inv, s_cnt, s_off, s_wsum);
}

// --------------------------------------------------------- k_route_decode
// Router row e (bf16 weights) against every token: logits[t][e] (+ bias).
template <int MC>
__device__ void router_row(const uint16_t* wrow, const uint16_t* x, int T, int H, float bias,
                           float* logits, int ldl, int e, int lane) {
    const int NC = H >> 5;
    uint4 wv[MC][4];
#pragma unroll
    for (int m = 0; m < MC; ++m)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int c = lane + 32 * m;
            wv[m][v] = (c < NC) ? ldg_stream(wrow + 32 * c + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
        }
    for (int t = 0; t < T; ++t) {
        uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
        for (int m = 0; m < MC; ++m) {
            const int c = lane + 32 * m;
            if (c < NC) {
                const uint4* xp = reinterpret_cast<const uint4*>(x + size_t(t) * H + 32 * c);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 xu = ldg_keep(xp + v);
                    const uint32_t xw[4] = {xu.x, xu.y, xu.z, xu.w};
                    const uint32_t ww[4] = {wv[m][v].x, wv[m][v].y, wv[m][v].z, wv[m][v].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint64_t a = pk(bf16_lo(ww[i]), bf16_hi(ww[i]));
                        const uint64_t b = pk(bf16_lo(xw[i]), bf16_hi(xw[i]));
                        if (i & 1)
                            acc1 = ffma2(a, b, acc1);
                        else
                            acc0 = ffma2(a, b, acc0);
                    }
                }
            }
        }
        const float2 a0 = upk(acc0), a1 = upk(acc1);
        const float sum = warp_sum((a0.x + a0.y) + (a1.x + a1.y));
        if (lane == 0) logits[size_t(t) * ldl + e] = sum + bias;
    }
}

// Top-K of one token's logits (larger first, ties to the lower id), stored
// in ascending id with renormalised softmax weights.  One warp; L is this
// warp's shared-memory copy of the logits.
__device__ void select_token(const RouteLaunch& a, int t, int lane, float* L, int32_t* s_ids) {
    const int E = a.E, K = a.K, ldl = E + 1;
    const float* lg = a.logits + size_t(t) * ldl;
    for (int e = lane; e < E; e += 32) L[e] = __ldcg(lg + e);
    __syncwarp();
    float selv[kMaxTopK];
    int sele[kMaxTopK];
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
        selv[k] = 0.0f;
        sele[k] = 0x7fffffff;
        if (k < K) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
            for (int e = lane; e < E; e += 32) {
                const float v = L[e];
                if (v > bv || (v == bv && e < be)) {
                    bv = v;
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (ov > bv || (ov == bv && oe < be)) {
                    bv = ov;
                    be = oe;
                }
            }
            selv[k] = bv;
            sele[k] = be;
            if (be < E && lane == (be & 31)) L[be] = __int_as_float(0x7fc00000);  // taken
            __syncwarp();
        }
    }
    // rank of each pick in ascending id
    int rank[kMaxTopK];
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
        int r = 0;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) r += (j < K && sele[j] < sele[k]) ? 1 : 0;
        rank[k] = r;
    }
    const float m = selv[0];
    float sum = 0.0f;
    for (int r = 0; r < K; ++r) {
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
            if (k < K && rank[k] == r) sum += expf(selv[k] - m);
    }
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
        if (k < K && rank[k] == lane) {
            const int id = sele[k];
            const float wv = expf(selv[k] - m) / sum;
            const size_t o = size_t(t) * K + lane;
            a.ids[o] = id;
            a.w[o] = wv;
            if (a.ids_user) a.ids_user[o] = id;
            if (a.w_user) a.w_user[o] = wv;
            s_ids[o] = id;
        }
    }
    if (a.logits_user)
        for (int e = lane; e < E; e += 32) a.logits_user[size_t(t) * E + e] = __ldcg(lg + e);
}

template <int MC, int RB>
__global__ void __launch_bounds__(256, 1) k_route_decode(RouteLaunch a) {
    extern __shared__ float s_dyn[];           // [warps][E] logits for selection
    __shared__ int s_last;
    __shared__ int32_t s_ids[kDecodeMaxTokens * kMaxTopK];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_wsum[32];
    Ctl* ctl = reinterpret_cast<Ctl*>(a.ctl);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, wpb = blockDim.x >> 5;
    const int ldl = a.E + 1;
    const int n_router = a.do_select ? a.E + 1 : 1;
    const int n_sh = a.do_shared ? (a.Is + RB - 1) / RB : 0;
    const int ntask = n_router + n_sh;

    for (int task = blockIdx.x + gridDim.x * wid; task < ntask; task += gridDim.x * wpb) {
        if (task < n_router) {
            const int e = a.do_select ? task : a.E;
            const float b = (e < a.E && a.bias) ? __ldg(a.bias + e) : 0.0f;
            router_row<MC>(a.router + size_t(e) * a.H, a.x, a.T, a.H, b, a.logits, ldl, e, lane);
        } else {
            const int i0 = (task - n_router) * RB;
            gu_batch<MC, RB>(a.shq, a.shs, a.H, i0, min(RB, a.Is - i0), a.x, 0, a.T, nullptr, 1,
                             a.T, a.hs, a.Is, &ctl->err, lane);
        }
    }

    // Last CTA to finish continues (no CTA waits for another).
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&ctl->arrive, 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    const int T = a.T, K = a.K, E = a.E;
    for (int t = wid; t < T; t += wpb) {
        if (a.do_select) {
            select_token(a, t, lane, s_dyn + size_t(wid) * E, s_ids);
        } else {
            for (int k = lane; k < K; k += 32) {
                const size_t o = size_t(t) * K + k;
                const int id = __ldg(a.ids_in + o);
                const float wv = __ldg(a.w_in + o);
                if (id < 0 || id >= E) latch(&ctl->err, STRATA_EBADROUTE);
                a.ids[o] = id;
                a.w[o] = wv;
                s_ids[o] = id;
            }
        }
        if (lane == 0) {
            const float s = 1.0f / (1.0f + expf(-__ldcg(a.logits + size_t(t) * ldl + E)));
            a.sig[t] = s;
            if (a.sig_user) a.sig_user[t] = s;
        }
    }
    __syncthreads();

    if (a.do_permute)
        permute_block(s_ids, T, K, E, a.counts, a.offsets, a.perm, a.inv, s_cnt, s_off, s_wsum);
    if (tid == 0) atomicExch(&ctl->arrive, 0u);
}

// ----------------------------------------------------------------- k_down
constexpr int kDownMaxRowsPerLane = kDownRowsPerCta;

__global__ void __launch_bounds__(384, 1) k_down(DownLaunch a) {
    extern __shared__ float s_y[];          // [(T*K + T)][kDownRowsPerCta]
    __shared__ ActiveList s_act;
    constexpr int RBc = kDownRowsPerCta;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, wpb = blockDim.x >> 5;
    const int o0 = blockIdx.x * RBc;
    const int nrow = min(RBc, a.H - o0);
    const int TK = a.T * a.K;
    const int nslot = TK + a.T;
    for (int i = tid; i < nslot * RBc; i += blockDim.x) s_y[i] = 0.0f;
    if (a.mode != kDownCombine) {
        build_active(s_act, a.offsets, a.E, TK, a.err);
    } else {
        if (tid == 0) s_act.n = 0;
        __syncthreads();
    }
    const int n_routed = s_act.n;
    const int n_units = n_routed + (a.mode != kDownSlots ? 1 : 0);

    for (int u = wid; u < n_units; u += wpb) {
        const uint8_t* qe;
        const uint16_t* se;
        const float* hb;
        int len, s0, scount, ybase;
        if (u < n_routed) {
            const int e = s_act.e[u];
            len = a.I;
            qe = a.q + size_t(e) * a.H * (size_t(a.I) >> 1);
            se = a.sc + size_t(e) * a.H * (size_t(a.I) >> 5);
            s0 = s_act.off[u];
            scount = s_act.cnt[u];
            hb = a.h;
            ybase = 0;
        } else {
            len = a.Is;
            qe = a.shq;
            se = a.shs;
            s0 = 0;
            scount = a.T;
            hb = a.hs;
            ybase = TK;
        }
        const int NCd = len >> 5;               // chunks per row (power of two <= 32)
        const int RPW = 32 / NCd;               // rows per warp pass
        const int c = lane & (NCd - 1), rs = lane / NCd;
        const int nr = (nrow > rs) ? (nrow - rs + RPW - 1) / RPW : 0;
        const size_t qrow = size_t(len) >> 1, srow = size_t(len) >> 5;
        uint4 qv[kDownMaxRowsPerLane];
        float sc[kDownMaxRowsPerLane];
#pragma unroll
        for (int m = 0; m < kDownMaxRowsPerLane; ++m) {
            if (m < nr) {
                const size_t row = size_t(o0 + rs + m * RPW);
                qv[m] = ldg_stream(qe + row * qrow + size_t(c) * 16);
                sc[m] = f16_to_f32(ldg_u16(se + row * srow + c));
            } else {
                qv[m] = make_uint4(0u, 0u, 0u, 0u);
                sc[m] = 0.0f;
            }
        }
        for (int si = 0; si < scount; ++si) {
            const int s = s0 + si;
            const float* hp = hb + size_t(s) * len + 32 * c;
            uint64_t x2[16];
            float X = 0.0f;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 f = ldcg_f4(hp + 4 * v);
                x2[2 * v] = pk(f.x, f.y);
                x2[2 * v + 1] = pk(f.z, f.w);
                X += (f.x + f.y) + (f.z + f.w);
            }
#pragma unroll
            for (int m = 0; m < kDownMaxRowsPerLane; ++m) {
                float part = 0.0f;
                if (m < nr) part = group_dot(dot_chunk(qv[m], x2), X, sc[m]);
                if (m < (RBc + RPW - 1) / RPW || m < nr) {
                    part = group_sum(part, NCd);
                    if (c == 0 && m < nr) s_y[size_t(ybase + s) * RBc + rs + m * RPW] = part;
                }
            }
        }
    }
    __syncthreads();

    if (a.mode == kDownSlots) {
        for (int i = tid; i < TK * nrow; i += blockDim.x) {
            const int s = i / nrow, r = i - s * nrow;
            a.y_out[size_t(s) * a.H + o0 + r] = f32_to_bf16(s_y[size_t(s) * RBc + r]);
        }
        return;
    }
    for (int i = tid; i < a.T * nrow; i += blockDim.x) {
        const int t = i / nrow, r = i - t * nrow, o = o0 + r;
        float acc = 0.0f;
        for (int k = 0; k < a.K; ++k) {
            const int sl = __ldcg(a.inv + size_t(t) * a.K + k);
            if (sl < 0 || sl >= TK) continue;
            const float yv = (a.mode == kDownFused)
                                 ? s_y[size_t(sl) * RBc + r]
                                 : __uint_as_float(uint32_t(__ldg(a.y_in + size_t(sl) * a.H + o))
                                                   << 16);
            acc += __ldcg(a.w + size_t(t) * a.K + k) * yv;
        }
        const float v = acc + __ldcg(a.sig + t) * s_y[size_t(TK + t) * RBc + r];
        const uint16_t ob = f32_to_bf16(v);
        a.out[size_t(t) * a.H + o] = ob;
        if (a.resid) a.resid[size_t(t) * a.H + o] += __uint_as_float(uint32_t(ob) << 16);
    }
}

// --------------------------------------------------------------- RMSNorm
__global__ void k_rmsnorm(const float* r, int T, int H, float eps, uint16_t* x) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* rt = r + size_t(t) * H;
    float ss = 0.0f;
    for (int h = lane * 4; h < H; h += 128) {
        const float4 v = *reinterpret_cast<const float4*>(rt + h);
        ss += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
    }
    ss = warp_sum(ss);
    const float denom = sqrtf(ss / float(H) + eps);
    for (int h = lane * 4; h < H; h += 128) {
        const float4 v = *reinterpret_cast<const float4*>(rt + h);
        const uint32_t p0 = uint32_t(f32_to_bf16(v.x / denom)) |
                            (uint32_t(f32_to_bf16(v.y / denom)) << 16);
        const uint32_t p1 = uint32_t(f32_to_bf16(v.z / denom)) |
                            (uint32_t(f32_to_bf16(v.w / denom)) << 16);
        *reinterpret_cast<uint2*>(x + size_t(t) * H + h) = make_uint2(p0, p1);
    }
}

// -------------------------------------------------------------- launchers
template <int MC, int RB>
static cudaError_t route_mc(const RouteLaunch& a, cudaStream_t s, int grid) {
    // 8 warps x E logits (<= 32 KB): within the default dynamic limit
    const size_t dyn = size_t(8) * a.E * sizeof(float);
    k_route_decode<MC, RB><<<grid, 256, dyn, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_route_decode(const RouteLaunch& a, cudaStream_t s) {
    const Dev d = device_info();
    const int grid = d.sms;
    const int mc = (a.H + 1023) / 1024;
    if (mc <= 1) return route_mc<1, 4>(a, s, grid);
    if (mc <= 2) return route_mc<2, 4>(a, s, grid);
    return route_mc<4, 2>(a, s, grid);
}

cudaError_t launch_gate_up_decode(const GuLaunch& a, cudaStream_t s) {
    const Dev d = device_info();
    const int mc = (a.H + 1023) / 1024;
    if (mc <= 1)
        k_gate_up<1, 4><<<d.sms, 256, 0, s>>>(a);
    else if (mc <= 2)
        k_gate_up<2, 4><<<d.sms, 256, 0, s>>>(a);
    else
        k_gate_up<4, 2><<<d.sms, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_down_decode(const DownLaunch& a, cudaStream_t s) {
    const int grid = (a.H + kDownRowsPerCta - 1) / kDownRowsPerCta;
    // (T*K + T) slots x 14 rows of fp32 (<= 30 KB): within the default dynamic limit
    const size_t dyn = size_t(a.T * a.K + a.T) * kDownRowsPerCta * sizeof(float);
    k_down<<<grid, 384, dyn, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_permute_small(const int32_t* ids, int T, int K, int E, int32_t* counts,
                                 int32_t* offsets, int32_t* perm, int32_t* inv, uint32_t* err,
                                 cudaStream_t s) {
    k_permute_small<<<1, 256, 0, s>>>(ids, T, K, E, counts, offsets, perm, inv, err);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float* r, int T, int H, float eps, uint16_t* x, cudaStream_t s) {
    const int warps = 8;
    k_rmsnorm<<<(T + warps - 1) / warps, warps * 32, 0, s>>>(r, T, H, eps, x);
    return cudaGetLastError();
}

}  // namespace strata
