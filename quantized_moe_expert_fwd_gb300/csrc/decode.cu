// decode.cu -- the decode-size (T <= 32) kernels of the routed MoE FFN.
//
// Three launches make one layer (Strata, "Qwen3.6-35B-A3B: pictures, several
// requests at once and speed", section "Speed": router top-k and grouping in
// one launch, the router and the shared gate in one product, shared
// gate+up+SwiGLU in one launch, the MoE end in one launch; PolyStrata,
// "Models and backends", section "What was tuned": a call's experts go
// through one launch per stage, and one launch adds them up):
//
//   k_route    router rows (E+1 of them: the last is the shared-expert gate)
//              and the shared expert's gate/up rows, spread over every SM:
//              logits and the shared SwiGLU vectors.
//   k_gate_up  every CTA first selects each token's top-K from the logits,
//              computes the renormalised softmax weights and the sigmoid gate
//              and buckets the (token, k) pairs by expert -- the same result
//              in every CTA, so no CTA waits for another; CTA 0 publishes it.
//              Then every touched expert's gate/up rows, each read once for
//              all tokens routed to it, SwiGLU in the epilogue.
//   k_down     for a block of output rows: every touched expert's down rows
//              and the shared expert's, then the weighted combine (or, as
//              separate calls, per-slot outputs / the combine of given
//              per-slot outputs).
//
// k_gate_up and k_down stream weights through shared-memory rings: one
// producer thread issues 1-D bulk copies (cp.async.bulk) that complete on
// mbarriers, consumer warps compute from shared memory and release the
// stage.  All three kernels chain with programmatic dependent launch: each
// triggers its dependents at once and touches nothing the previous kernel
// writes before griddepcontrol.wait; weights that do not depend on routing
// (router rows, shared-expert rows) are requested before that wait.
// int4 weights become fp32 by byte placement (common.cuh); every sum has a
// fixed order, so results do not depend on timing.

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "route.cuh"

namespace strata {

// ---------------------------------------------------------------- k_route
template <int MC>
struct RouterRow {
    uint4 w[MC][4];
};

template <int MC>
__device__ __forceinline__ void router_load(RouterRow<MC>& R, const uint16_t* wrow, int H,
                                            int lane) {
    const int NC = H >> 5;
#pragma unroll
    for (int m = 0; m < MC; ++m)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int c = lane + 32 * m;
            R.w[m][v] = (c < NC) ? ldg_stream(wrow + 32 * c + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
        }
}

// logits[t][e] = router row e . x[t] (+ bias), every token.  One warp.
template <int MC>
__device__ void router_compute(const RouterRow<MC>& R, const uint16_t* x, int T, int H,
                               float bias, float* logits, int ldl, int e, int lane) {
    const int NC = H >> 5;
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
                    const uint32_t ww[4] = {R.w[m][v].x, R.w[m][v].y, R.w[m][v].z, R.w[m][v].w};
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

// Registers of RB gate/up row pairs of the shared expert (k_route's share).
template <int MC, int RB>
struct GuRows {
    uint4 q[RB][2][MC];
    float s[RB][2][MC];
};

template <int MC, int RB>
__device__ __forceinline__ void gu_load(GuRows<MC, RB>& R, const uint8_t* qe, const uint16_t* se,
                                        int H, int i0, int nb, int lane) {
    const int NC = H >> 5;
    const size_t qrow = size_t(H) >> 1, srow = size_t(H) >> 5;
#pragma unroll
    for (int p = 0; p < RB; ++p)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int m = 0; m < MC; ++m) {
                const int c = lane + 32 * m;
                const size_t row = size_t(2 * (i0 + p) + r);
                if (p < nb && c < NC) {
                    R.q[p][r][m] = ldg_stream(qe + row * qrow + size_t(c) * 16);
                    R.s[p][r][m] = f16_to_f32(ldg_u16(se + row * srow + c));
                } else {
                    R.q[p][r][m] = make_uint4(0u, 0u, 0u, 0u);
                    R.s[p][r][m] = 0.0f;
                }
            }
}

// hs[t][i0 + p] = silu(g) u for every token, row pairs p < nb.  One warp.
template <int MC, int RB>
__device__ void gu_compute_all_tokens(const GuRows<MC, RB>& R, int H, int T, int i0, int nb,
                                      const uint16_t* x, float* h, int ldh, int lane) {
    const int NC = H >> 5;
    for (int t = 0; t < T; ++t) {
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
                        a += group_dot(dot_chunk(R.q[p][r][m], x2[m]), X[m], R.s[p][r][m]);
                acc[p][r] = warp_sum(a);
            }
        float g = 0.0f, u = 0.0f;
#pragma unroll
        for (int p = 0; p < RB; ++p)
            if (p == lane) {
                g = acc[p][0];
                u = acc[p][1];
            }
        if (lane < nb) h[size_t(t) * ldh + i0 + lane] = silu_mul(g, u);
    }
}

template <int MC, int RB>
__global__ void __launch_bounds__(256, 1) k_route(RouteLaunch a) {
    pdl_launch();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, wpb = blockDim.x >> 5;
    const int ldl = a.E + 1;
    const int n_router = a.do_select ? a.E + 1 : 1;
    const int n_sh = a.do_shared ? (a.Is + RB - 1) / RB : 0;
    const int ntask = n_router + n_sh;
    // The first task's weights do not depend on the previous kernel: they are
    // requested before waiting for it.
    bool waited = false;
    for (int task = blockIdx.x + gridDim.x * wid; task < ntask; task += gridDim.x * wpb) {
        if (task < n_router) {
            const int e = a.do_select ? task : a.E;
            RouterRow<MC> R;
            router_load<MC>(R, a.router + size_t(e) * a.H, a.H, lane);
            const float b = (e < a.E && a.bias) ? __ldg(a.bias + e) : 0.0f;
            if (!waited) pdl_wait();
            waited = true;
            router_compute<MC>(R, a.x, a.T, a.H, b, a.logits, ldl, e, lane);
        } else {
            const int i0 = (task - n_router) * RB;
            const int nb = min(RB, a.Is - i0);
            GuRows<MC, RB> R;
            gu_load<MC, RB>(R, a.shq, a.shs, a.H, i0, nb, lane);
            if (!waited) pdl_wait();
            waited = true;
            gu_compute_all_tokens<MC, RB>(R, a.H, a.T, i0, nb, a.x, a.hs, a.Is, lane);
        }
    }
    if (!waited) pdl_wait();
}

// The routing of moe_route: one CTA selects every token (T <= 32) from the
// logits k_route wrote.
__global__ void __launch_bounds__(256, 1) k_select(SelectLaunch a) {
    extern __shared__ float s_dyn[];
    __shared__ int s_ids[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_w[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_sig[kDecodeMaxTokens];
    pdl_launch();
    pdl_wait();
    route_cta(a.logits, a.T, a.E, a.K, nullptr, nullptr, s_ids, s_w, s_sig, s_dyn, a.err,
              int(threadIdx.x), int(blockDim.x), BlockSync{});
    const int TK = a.T * a.K;
    for (int p = threadIdx.x; p < TK; p += blockDim.x) {
        a.ids[p] = s_ids[p];
        a.w[p] = s_w[p];
    }
    for (int t = threadIdx.x; t < a.T; t += blockDim.x) a.sig[t] = s_sig[t];
    if (a.logits_out)
        for (int i = threadIdx.x; i < a.T * a.E; i += blockDim.x)
            a.logits_out[i] = __ldcg(a.logits + size_t(i / a.E) * (a.E + 1) + i % a.E);
}

// -------------------------------------------------------------- bucketing
// Standalone bucketing of up to kDecodeMaxTokens * kMaxTopK pairs.
__global__ void __launch_bounds__(256, 1) k_permute_small(const int32_t* ids, int T, int K, int E,
                                                          int32_t* counts, int32_t* offsets,
                                                          int32_t* perm, int32_t* inv,
                                                          uint32_t* err) {
    __shared__ int s_ids[kDecodeMaxTokens * kMaxTopK];
    __shared__ int s_inv[kDecodeMaxTokens * kMaxTopK];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_wsum[32];
    __shared__ SPlan P;
    pdl_launch();
    pdl_wait();
    for (int p = threadIdx.x; p < T * K; p += blockDim.x) {
        const int e = __ldg(ids + p);
        if (e < 0 || e >= E) latch(err, STRATA_EBADROUTE);
        s_ids[p] = e;
    }
    __syncthreads();
    const BucketOut g{counts, offsets, perm, inv, nullptr};
    bucket_cta(s_ids, T, K, E, s_cnt, s_off, s_wsum, P, s_inv, g, int(threadIdx.x),
               int(blockDim.x), BlockSync{});
}

// The plan from a bucketing given by the caller (offsets and perm from any
// source); inconsistent entries latch STRATA_EBADROUTE and are left out.
__global__ void __launch_bounds__(256, 1) k_plan(const int32_t* offsets, const int32_t* perm,
                                                 int T, int K, int E, int32_t* plan,
                                                 uint32_t* err) {
    __shared__ int warp_base[32];
    __shared__ int running;
    pdl_launch();
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    const int TK = T * K;
    // token of each slot; without perm (the down product needs slots only) 0
    for (int s = tid; s < TK; s += blockDim.x) {
        int t = 0;
        if (perm != nullptr) {
            const int p = __ldg(perm + s);
            if (p >= 0 && p < TK) {
                t = p / K;
            } else {
                latch(err, STRATA_EBADROUTE);
                t = -1;
            }
        }
        plan[kPlanHeader + 3 * E + s] = t;
    }
    if (tid == 0) running = 0;
    __syncthreads();
    for (int base = 0; base < E; base += blockDim.x) {
        const int e = base + tid;
        int off = 0, cnt = 0;
        if (e < E) {
            off = __ldg(offsets + e);
            const int end = __ldg(offsets + e + 1);
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
            plan[kPlanHeader + pos] = e;
            plan[kPlanHeader + E + pos] = off;
            plan[kPlanHeader + 2 * E + pos] = cnt;
        }
        __syncthreads();
    }
    if (tid == 0) plan[0] = running;
}

// -------------------------------------------------------------- k_gate_up
// Consumer warps and row pairs per ring stage.  A stage holds kGuRowPairs
// interleaved gate/up row pairs of one expert (their packed bytes and their
// scales, two bulk copies); consumer warp w computes row pairs w and
// w + kGuConsumers of every stage.
constexpr int kGuConsumers = 8;
constexpr int kGuRowPairs = 16;
constexpr int kGuThreads = 32 * (kGuConsumers + 1);

template <int MC>
__global__ void __launch_bounds__(kGuThreads, 1) k_gate_up(GuLaunch a) {
    extern __shared__ __align__(128) uint8_t g_ring[];
    __shared__ SPlan P;
    __shared__ int s_ids[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_w[kDecodeMaxTokens * kMaxTopK];
    __shared__ int s_inv[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_sig[kDecodeMaxTokens];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_wsum[32];
    __shared__ __align__(8) uint64_t full[kGuMaxStages], empty[kGuMaxStages];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int S = a.stages;
    pdl_launch();
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kGuConsumers);
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();

    const int T = a.T, K = a.K, E = a.E, H = a.H, I = a.I;
    if (a.mode == kGuShared) {
        shared_plan(P, T);
    } else if (a.mode == kGuPlan) {
        load_plan(P, a.plan, E, T * K);
    } else {
        // routing: the same in every CTA; CTA 0 publishes it
        route_cta(a.logits, T, E, K, a.forced_ids, a.forced_w, s_ids, s_w, s_sig,
                  reinterpret_cast<float*>(g_ring), a.err, tid, int(blockDim.x), BlockSync{});
        // tail-skip: the bucketing sees the left-out picks as unrouted; the
        // selection's scratch at the start of the ring is free until the
        // first weight copy, which needs the plan
        const int* bids = s_ids;
        if (a.tail_skip > 0 && a.tail_skip < K) {
            int* rank = reinterpret_cast<int*>(g_ring);
            int* bid = rank + kDecodeMaxTokens * kMaxTopK;
            int* keep = bid + kDecodeMaxTokens * kMaxTopK;
            tail_skip_cta(s_ids, s_w, T, K, E, a.tail_skip, rank, bid, keep, tid,
                          int(blockDim.x));
            bids = bid;
        }
        // the plan only; CTA 0 publishes the routing and the bucketing after
        // its share of the experts, off the path to the first weight copy
        const BucketOut none{nullptr, nullptr, nullptr, nullptr, nullptr};
        bucket_cta(bids, T, K, E, s_cnt, s_off, s_wsum, P, s_inv, none, tid, int(blockDim.x),
                   BlockSync{});
        __syncthreads();
    }

    // this CTA's contiguous share of the touched experts' row pairs, cut by
    // cost: a row pair of expert j costs its tokens plus one (the read of
    // its rows), so CTAs on an expert with many tokens take fewer of its rows
    auto rp_at = [&](long long x) {
        long long cum = 0;
        for (int j = 0; j < P.n; ++j) {
            const long long w = (long long)P.cnt[j] + 1, cj = w * I;
            if (x < cum + cj) return (long long)j * I + (x - cum) / w;
            cum += cj;
        }
        return (long long)P.n * I;
    };
    long long cost = 0;
    for (int j = 0; j < P.n; ++j) cost += ((long long)P.cnt[j] + 1) * I;
    const long long beg = rp_at((long long)blockIdx.x * cost / gridDim.x);
    const long long end = rp_at((long long)(blockIdx.x + 1) * cost / gridDim.x);
    const size_t qrow = size_t(H) >> 1, srow = size_t(H) >> 5;   // bytes, scales per row
    const size_t qexp = size_t(2) * I * qrow, sexp = size_t(2) * I * srow;
    const uint32_t stage_q = uint32_t(kGuRowPairs * 2 * qrow);
    const uint32_t stage_bytes = stage_q + uint32_t(kGuRowPairs * 2 * srow * 2);

    if (wid == 0) {
        // producer
        if (lane == 0) {
            int i = 0;
            for (long long rp = beg; rp < end; ++i) {
                const int j = int(rp / I), i0 = int(rp % I);
                const int nb = int(min((long long)kGuRowPairs, min((long long)(I - i0), end - rp)));
                const int slot = i % S, round = i / S;
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1))
                    latch_timeout(a.err, 1, slot, round, i);
                const int e = P.e[j];
                uint8_t* dq = g_ring + size_t(slot) * stage_bytes;
                const uint32_t bq = uint32_t(nb * 2 * qrow), bs = uint32_t(nb * 2 * srow * 2);
                mbar_expect_tx(&full[slot], bq + bs);
                bulk_g2s(dq, a.q + size_t(e) * qexp + size_t(2 * i0) * qrow, bq, &full[slot]);
                bulk_g2s(dq + stage_q, a.sc + size_t(e) * sexp + size_t(2 * i0) * srow, bs,
                         &full[slot]);
                rp += nb;
            }
        }
        return;
    }

    // consumers: first (x_smem) every token's activations into shared memory
    // after the ring, chunk-interleaved, while the producer's first copies fly
    const int cw = wid - 1;
    const int NC = H >> 5;
    uint64_t x2[MC][16];
    float X[MC];
    uint4* xs = reinterpret_cast<uint4*>(g_ring + size_t(S) * stage_bytes);
    if (a.x_smem) {
        for (int i = tid - 32; i < T * 4 * NC; i += kGuConsumers * 32) {
            const int t = i / (4 * NC), r = i - t * 4 * NC, c = r >> 2, v = r & 3;
            xs[size_t(t) * 4 * NC + v * NC + c] =
                ldg_keep(reinterpret_cast<const uint4*>(a.x + size_t(t) * H) + 4 * c + v);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kGuConsumers * 32) : "memory");
    }
    // token t's activations into x2 / X
    auto get_x = [&](int t) {
        if (a.x_smem)
            load_x_smem<MC>(xs + size_t(t) * 4 * NC, NC, lane, x2, X);
        else
            load_x<MC>(a.x + size_t(t) * H, NC, lane, x2, X);
    };
    int xt = -1;              // token whose activations x2 holds
    int i = 0;
    for (long long rp = beg; rp < end; ++i) {
        const int j = int(rp / I), i0 = int(rp % I);
        const int nb = int(min((long long)kGuRowPairs, min((long long)(I - i0), end - rp)));
        const int slot = i % S, round = i / S;
        const int s0 = P.off[j], scount = P.cnt[j];
        if (scount > 0 && P.tok[s0] != xt && P.tok[s0] >= 0 && P.tok[s0] < T) {
            xt = P.tok[s0];
            get_x(xt);                 // overlaps the copy
        }
        if (!mbar_wait(&full[slot], round & 1)) latch_timeout(a.err, 2, slot, round, i);
        const uint8_t* sq = g_ring + size_t(slot) * stage_bytes;
        const uint16_t* ss = reinterpret_cast<const uint16_t*>(sq + stage_q);
        for (int si = 0; si < scount; ++si) {
            const int s = s0 + si;
            const int t = P.tok[s];
            if (t < 0 || t >= T) continue;
            if (t != xt) {
                xt = t;
                get_x(t);
            }
#pragma unroll
            for (int pp = 0; pp < kGuRowPairs / kGuConsumers; ++pp) {
                const int p = cw + pp * kGuConsumers;
                if (p >= nb) break;
                float acc[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint8_t* qr = sq + size_t(2 * p + r) * qrow;
                    const uint16_t* sr = ss + size_t(2 * p + r) * srow;
                    float v = 0.0f;
#pragma unroll
                    for (int m = 0; m < MC; ++m) {
                        const int c = lane + 32 * m;
                        if (c < NC) {
                            const uint4 q = *reinterpret_cast<const uint4*>(qr + 16 * c);
                            const float sc = f16_to_f32(sr[c]);
                            v += group_dot(dot_chunk(q, x2[m]), X[m], sc);
                        }
                    }
                    acc[r] = warp_sum(v);
                }
                if (lane == 0) a.h[size_t(s) * I + i0 + p] = silu_mul(acc[0], acc[1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        rp += nb;
    }
    if (a.mode == kGuRoute && blockIdx.x == 0) {
        const int ct = tid - 32, cn = kGuConsumers * 32;
        publish_bucket(T * K, E, P, s_inv,
                       BucketOut{a.counts, a.offsets, a.perm, a.inv, a.plan_out}, ct, cn);
        for (int p = ct; p < T * K; p += cn) {
            a.ids[p] = s_ids[p];
            a.w[p] = s_w[p];
            if (a.ids_user) a.ids_user[p] = s_ids[p];
            if (a.w_user) a.w_user[p] = s_w[p];
        }
        for (int t = ct; t < T; t += cn) {
            a.sig[t] = s_sig[t];
            if (a.sig_user) a.sig_user[t] = s_sig[t];
        }
    }
}

// ----------------------------------------------------------------- k_down
// A CTA owns kDownRowsPerCta output rows.  Ring stages hold one expert's
// slice of those rows (packed bytes and scales, two bulk copies); consumer
// warp w computes the units w, w + kDnConsumers, ...: unit 0 is the shared
// expert (its copy is requested before griddepcontrol.wait), units 1.. the
// touched experts.  Lane (rs, c) of a warp holds chunk c of rows rs,
// rs + RPW, ... (RPW = 32 / chunks per row).
constexpr int kDnConsumers = 12;
constexpr int kDnThreads = 32 * (kDnConsumers + 1);
static_assert(kDnMaxStages % kDnConsumers == 0, "stages must be a multiple of consumer warps");

template <int MR>
__device__ void down_unit(const uint8_t* sq, const uint16_t* ss, int len, int nrow, int lane,
                          const float* hb, int s0, int scount, const int* tok, float* s_y,
                          int ybase) {
    constexpr int RBc = kDownRowsPerCta;
    const int NCd = len >> 5, RPW = 32 / NCd;
    const int c = lane & (NCd - 1), rs = lane / NCd;
    const int nr = (nrow > rs) ? (nrow - rs + RPW - 1) / RPW : 0;
    const int npass = (RBc + RPW - 1) / RPW;     // uniform over the warp
    const size_t qrow = size_t(len) >> 1, srow = size_t(len) >> 5;
    uint4 q[MR];
    float sc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
        if (m < nr) {
            const int row = rs + m * RPW;
            q[m] = *reinterpret_cast<const uint4*>(sq + row * qrow + 16 * c);
            sc[m] = f16_to_f32(ss[row * srow + c]);
        } else {
            q[m] = make_uint4(0u, 0u, 0u, 0u);
            sc[m] = 0.0f;
        }
    }
    for (int si = 0; si < scount; ++si) {
        const int s = s0 + si;
        if (tok != nullptr && tok[s] < 0) continue;
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
        for (int m = 0; m < MR; ++m) {
            if (m < npass) {
                float part = (m < nr) ? group_dot(dot_chunk(q[m], x2), X, sc[m]) : 0.0f;
                part = group_sum(part, NCd);
                if (c == 0 && m < nr) s_y[size_t(ybase + s) * RBc + rs + m * RPW] = part;
            }
        }
    }
}

template <int MR>
__global__ void __launch_bounds__(kDnThreads, 1) k_down(DownLaunch a) {
    extern __shared__ __align__(128) uint8_t d_dyn[];
    __shared__ SPlan P;
    __shared__ int s_inv[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_w[kDecodeMaxTokens * kMaxTopK];
    __shared__ float s_sig[kDecodeMaxTokens];
    __shared__ __align__(8) uint64_t full[kDnMaxStages], empty[kDnMaxStages];
    constexpr int RBc = kDownRowsPerCta;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int S = a.stages;
    const int o0 = blockIdx.x * RBc;
    const int nrow = min(RBc, a.H - o0);
    const int TK = a.T * a.K;
    const bool with_shared = a.mode != kDownSlots;
    const int len = a.I > a.Is ? a.I : a.Is;
    const uint32_t stage_q = uint32_t(RBc * (len >> 1));
    const uint32_t stage_bytes = stage_q + uint32_t(RBc * (len >> 5) * 2);
    float* s_y = reinterpret_cast<float*>(d_dyn + size_t(S) * stage_bytes);

    // unit u's packed rows and scales: the shared expert is unit 0 when present
    auto issue = [&](int u, int slot, int e) {
        const bool sh = with_shared && u == 0;
        const int L = sh ? a.Is : a.I;
        const uint8_t* q = sh ? a.shq : a.q + size_t(e) * a.H * (size_t(L) >> 1);
        const uint16_t* sc = sh ? a.shs : a.sc + size_t(e) * a.H * (size_t(L) >> 5);
        const uint32_t bq = uint32_t(nrow * (L >> 1)), bs = uint32_t(nrow * (L >> 5) * 2);
        uint8_t* dst = d_dyn + size_t(slot) * stage_bytes;
        mbar_expect_tx(&full[slot], bq + bs);
        bulk_g2s(dst, q + size_t(o0) * (L >> 1), bq, &full[slot]);
        bulk_g2s(dst + stage_q, sc + size_t(o0) * (L >> 5), bs, &full[slot]);
    };

    pdl_launch();
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_fence_init();
        if (with_shared) issue(0, 0, 0);       // static weights: before the wait
    }
    __syncthreads();
    pdl_wait();

    for (int i = tid; i < (TK + a.T) * RBc; i += blockDim.x) s_y[i] = 0.0f;
    if (a.mode == kDownCombine) {
        if (tid == 0) P.n = 0;
    } else {
        load_plan(P, a.plan, a.E, TK);
    }
    if (a.mode != kDownSlots) {
        for (int i = tid; i < TK; i += blockDim.x) {
            s_inv[i] = __ldcg(a.inv + i);
            s_w[i] = __ldcg(a.w + i);
        }
        for (int t = tid; t < a.T; t += blockDim.x) s_sig[t] = __ldcg(a.sig + t);
    }
    __syncthreads();

    const int sh = with_shared ? 1 : 0;
    const int n_units = P.n + sh;
    if (wid == 0) {
        if (lane == 0) {
            for (int u = sh; u < n_units; ++u) {
                const int slot = u % S, round = u / S;
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1))
                    latch_timeout(a.err, 3, slot, round, u);
                issue(u, slot, P.e[u - sh]);
            }
        }
    } else {
        for (int u = wid - 1; u < n_units; u += kDnConsumers) {
            const int slot = u % S, round = u / S;
            if (!mbar_wait(&full[slot], round & 1)) latch_timeout(a.err, 4, slot, round, u);
            const uint8_t* sq = d_dyn + size_t(slot) * stage_bytes;
            const uint16_t* ss = reinterpret_cast<const uint16_t*>(sq + stage_q);
            if (with_shared && u == 0) {
                down_unit<MR>(sq, ss, a.Is, nrow, lane, a.hs, 0, a.T, nullptr, s_y, TK);
            } else {
                const int j = u - sh;
                down_unit<MR>(sq, ss, a.I, nrow, lane, a.h, P.off[j], P.cnt[j], P.tok, s_y, 0);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
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
            const int sl = s_inv[t * a.K + k];
            if (sl < 0 || sl >= TK) continue;
            const float yv = (a.mode == kDownFused)
                                 ? s_y[size_t(sl) * RBc + r]
                                 : __uint_as_float(uint32_t(__ldg(a.y_in + size_t(sl) * a.H + o))
                                                   << 16);
            acc += s_w[t * a.K + k] * yv;
        }
        const float v = acc + s_sig[t] * s_y[size_t(TK + t) * RBc + r];
        const uint16_t ob = f32_to_bf16(v);
        a.out[size_t(t) * a.H + o] = ob;
        if (a.resid) a.resid[size_t(t) * a.H + o] += __uint_as_float(uint32_t(ob) << 16);
    }
}

// --------------------------------------------------------------- RMSNorm
__global__ void k_rmsnorm(const float* r, int T, int H, float eps, uint16_t* x) {
    pdl_launch();
    pdl_wait();
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
// Every launch carries the programmatic-stream-serialization attribute, so a
// kernel may start while its predecessor on the stream drains; the kernels
// themselves wait (griddepcontrol.wait) before touching anything the
// predecessor writes.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem,
                              cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e == cudaSuccess) prof_after_launch(s);
    return e;
}

template <typename K>
static cudaError_t allow_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

cudaError_t launch_route_decode(const RouteLaunch& a, cudaStream_t s) {
    const Dev d = device_info();
    const int mc = (a.H + 1023) / 1024;
    if (mc <= 1) return launch_pdl(k_route<1, 4>, d.sms, 256, 0, s, a);
    if (mc <= 2) return launch_pdl(k_route<2, 4>, d.sms, 256, 0, s, a);
    return launch_pdl(k_route<4, 2>, d.sms, 256, 0, s, a);
}

cudaError_t launch_select(const SelectLaunch& a, cudaStream_t s) {
    const size_t dyn = size_t(8) * (a.E + 16) * sizeof(float);     // <= 33 KB
    return launch_pdl(k_select, 1, 256, dyn, s, a);
}

// Ring stages of k_gate_up: as many as kGuRingBytes holds, fewer when the T
// tokens' activations (T * H bf16 after the ring, x_smem) would not fit
// beside them; with fewer than two stages left the activations stay in
// global memory.
int gate_up_stages(int H, int T, int* x_smem) {
    const size_t stage = size_t(kGuRowPairs) * 2 * (size_t(H) / 2 + size_t(H) / 16);
    const size_t xbytes = size_t(T) * H * 2;
    size_t room = kGuSmemBytes > xbytes ? kGuSmemBytes - xbytes : 0;
    *x_smem = room >= 2 * stage ? 1 : 0;
    if (!*x_smem || room > kGuRingBytes) room = kGuRingBytes;
    const int S = int(room / stage);
    return S < kGuMaxStages ? S : kGuMaxStages;
}

cudaError_t launch_gate_up_decode(GuLaunch a, cudaStream_t s) {
    const Dev d = device_info();
    const int mc = (a.H + 1023) / 1024;
    a.stages = gate_up_stages(a.H, a.T, &a.x_smem);
    const size_t stage = size_t(kGuRowPairs) * 2 * (size_t(a.H) / 2 + size_t(a.H) / 16);
    size_t dyn = size_t(a.stages) * stage + (a.x_smem ? size_t(a.T) * a.H * 2 : 0);
    const size_t sel = size_t(kGuConsumers + 1) * (a.E + 16) * sizeof(float);
    if (dyn < sel) dyn = sel;
    // tail-skip scratch (ranks, bucketing ids, expert flags) at the ring's start
    const size_t skip = size_t(2 * kDecodeMaxTokens * kMaxTopK + a.E) * sizeof(int);
    if (a.tail_skip > 0 && dyn < skip) dyn = skip;
    cudaError_t err;
    if (mc <= 1) {
        if ((err = allow_smem(k_gate_up<1>, dyn)) != cudaSuccess) return err;
        return launch_pdl(k_gate_up<1>, d.sms, kGuThreads, dyn, s, a);
    }
    if (mc <= 2) {
        if ((err = allow_smem(k_gate_up<2>, dyn)) != cudaSuccess) return err;
        return launch_pdl(k_gate_up<2>, d.sms, kGuThreads, dyn, s, a);
    }
    if ((err = allow_smem(k_gate_up<4>, dyn)) != cudaSuccess) return err;
    return launch_pdl(k_gate_up<4>, d.sms, kGuThreads, dyn, s, a);
}

cudaError_t launch_down_decode(DownLaunch a, cudaStream_t s) {
    const int grid = (a.H + kDownRowsPerCta - 1) / kDownRowsPerCta;
    const int len = a.I > a.Is ? a.I : a.Is;
    const size_t stage = size_t(kDownRowsPerCta) * (size_t(len) / 2 + size_t(len) / 16);
    // A multiple of the consumer warps: unit u goes to warp u % kDnConsumers
    // and slot u % S, so every round of a slot belongs to one warp and its
    // parity waits never run ahead of the slot's phase.
    int S = int(kDnRingBytes / (stage * kDnConsumers)) * kDnConsumers;
    if (S < kDnConsumers) S = kDnConsumers;
    a.stages = S < kDnMaxStages ? S : (kDnMaxStages / kDnConsumers) * kDnConsumers;
    const size_t dyn = size_t(a.stages) * stage +
                       size_t(a.T * a.K + a.T) * kDownRowsPerCta * sizeof(float);
    // rows per lane: kDownRowsPerCta rows over 32 / (len / 32) row groups
    const int rpw = 1024 / len;
    const int mr = (kDownRowsPerCta + rpw - 1) / rpw;
    cudaError_t err;
#define STRATA_DOWN(MRV)                                                        \
    if ((err = allow_smem(k_down<MRV>, dyn)) != cudaSuccess) return err;        \
    return launch_pdl(k_down<MRV>, grid, kDnThreads, dyn, s, a)
    if (mr <= 1) { STRATA_DOWN(1); }
    if (mr <= 2) { STRATA_DOWN(2); }
    if (mr <= 4) { STRATA_DOWN(4); }
    if (mr <= 8) { STRATA_DOWN(8); }
    STRATA_DOWN(16);
#undef STRATA_DOWN
}

cudaError_t launch_plan(const int32_t* offsets, const int32_t* perm, int T, int K, int E,
                        int32_t* plan, uint32_t* err, cudaStream_t s) {
    return launch_pdl(k_plan, 1, 256, 0, s, offsets, perm, T, K, E, plan, err);
}

cudaError_t launch_permute_small(const int32_t* ids, int T, int K, int E, int32_t* counts,
                                 int32_t* offsets, int32_t* perm, int32_t* inv, uint32_t* err,
                                 cudaStream_t s) {
    return launch_pdl(k_permute_small, 1, 256, 0, s, ids, T, K, E, counts, offsets, perm, inv,
                      err);
}

cudaError_t launch_rmsnorm(const float* r, int T, int H, float eps, uint16_t* x, cudaStream_t s) {
    const int warps = 8;
    return launch_pdl(k_rmsnorm, (T + warps - 1) / warps, warps * 32, 0, s, r, T, H, eps, x);
}

}  // namespace strata
