// prefill.cu -- the large-T (prefill) path of the routed MoE FFN on the
// 5th-generation tensor cores: routing, bucketing, gathering and the
// combine (the expert GEMMs are in prefill_gemm.cu).
//
// The pages found the prompt path bound by "dequantize each expert to FP16
// and call oneMKL" (Strata, "Strata on an Intel Arc", section "The engine
// itself on Intel: the SYCL port") and by per-layer host grouping; a fused
// dequant + matrix-unit kernel lost there because it did not overlap the
// two.  Here every step runs on the GPU:
//
//   k_pf_router     K slices of logits = x * router^T (bf16 x bf16 -> fp32,
//                   tcgen05), one CTA a (expert tile, token tile, slice)
//   k_pf_select     slices added in order + bias; top-K, softmax weights,
//                   sigmoid gate: one warp a token
//   k_pf_count / k_pf_scan / k_pf_scatter
//                   stable counting sort of the (token, k) pairs by expert
//                   and the list of 128-row blocks of every expert ("a
//                   layer's cached experts in a few launches, by how many
//                   rows each has", PolyStrata, "Models and backends",
//                   section "What was tuned"); the shared expert is one more
//                   group whose rows are all tokens
//   k_pf_gather     activations of every slot, fp16, in the operand order
//   gate/up, down   grouped GEMMs with the dequantised int4 weights in TMEM
//                   (prefill_gemm.cu) -> h (fp16), y (fp16 or bf16)
//   k_pf_combine    out = sum_k w y + sigma(gate) S, in a fixed order
//
// Operand order inside each group of 8 along K: [0,4,1,5,2,6,3,7], the
// order in which the weight dequantisation yields its fp16 pairs; writing
// the activations in the same order makes the products the natural ones,
// since the MMA sums over K in any consistent order.

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "route.cuh"
#include "tc.cuh"

namespace strata {

// ------------------------------------------------------------- selection
// Token t's logits e = lane + 32 i (i < NR; e = E is the gate) into the
// warp's keys Lk and *gate: every K slice requested at once (one round trip),
// the slices added in slice order (slice 0 holds the bias).  NR = 0: E too large for
// registers, four logits a round.
template <int NR>
__device__ __forceinline__ void pf_logits(const PfSelectLaunch& a, int t, int lane, uint32_t* Lk,
                                          float* gate) {
    const int E = a.E, S = a.nsplit;
    const size_t ld = size_t(E) + 1, sstride = size_t(a.T) * ld;
    const float* p = a.part + size_t(t) * ld;
    if constexpr (NR > 0) {
        float u[kRouterSplitMax][NR];
#pragma unroll
        for (int sl = 0; sl < kRouterSplitMax; ++sl)
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                const int e = lane + 32 * i;
                u[sl][i] = (sl < S && e <= E) ? __ldcg(p + sl * sstride + e) : 0.0f;
            }
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int e = lane + 32 * i;
            float v = 0.0f;
#pragma unroll
            for (int sl = 0; sl < kRouterSplitMax; ++sl) v += u[sl][i];
            if (e < E) {
                Lk[e] = logit_key(v);
                if (a.logits_user) a.logits_user[size_t(t) * E + e] = v;
            } else if (e == E) {
                *gate = v;
            }
        }
    } else {
#pragma unroll 1
        for (int e0 = lane; e0 <= E; e0 += 4 * 32) {
            float u[kRouterSplitMax][4];
#pragma unroll
            for (int sl = 0; sl < kRouterSplitMax; ++sl)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    u[sl][j] = (sl < S && e0 + 32 * j <= E)
                                   ? __ldcg(p + sl * sstride + e0 + 32 * j)
                                   : 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = e0 + 32 * j;
                float v = 0.0f;
#pragma unroll
                for (int sl = 0; sl < kRouterSplitMax; ++sl) v += u[sl][j];
                if (e < E) {
                    Lk[e] = logit_key(v);
                    if (a.logits_user) a.logits_user[size_t(t) * E + e] = v;
                } else if (e == E) {
                    *gate = v;
                }
            }
        }
    }
}

// One warp a token: the logits are the router GEMM's K slices added in slice
// order (the bias is in slice 0); then top-K (ties to the lower id), ids ascending,
// renormalised softmax weights and the sigmoid of the shared-gate logit, by
// the decode path's selection; or the forced ids/weights.
template <int NR>
__global__ void __launch_bounds__(256) k_pf_select(PfSelectLaunch a) {
    extern __shared__ float s_dyn[];
    pdl_launch();
    pdl_wait();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int t = blockIdx.x * (blockDim.x >> 5) + wid;
    if (t >= a.T) return;
    const int E = a.E, K = a.K;
    float* L = s_dyn + size_t(wid) * (E + 16);
    uint32_t* Lk = reinterpret_cast<uint32_t*>(L);
    __shared__ int s_ids[8][kMaxTopK];
    __shared__ float s_w[8][kMaxTopK];
    __shared__ float s_gate[8];
    pf_logits<NR>(a, t, lane, Lk, &s_gate[wid]);
    __syncwarp();
    if (a.forced_ids) {
        for (int k = lane; k < K; k += 32) {
            const int id = __ldg(a.forced_ids + size_t(t) * K + k);
            if (id < 0 || id >= E) latch(a.err, STRATA_EBADROUTE);
            s_ids[wid][k] = id;
            s_w[wid][k] = __ldg(a.forced_w + size_t(t) * K + k);
        }
        __syncwarp();
    } else {
        select_topk_keys(E, K, Lk, L + E, s_ids[wid], s_w[wid], lane);
    }
    for (int k = lane; k < K; k += 32) {
        const size_t o = size_t(t) * K + k;
        a.ids[o] = s_ids[wid][k];
        a.w[o] = s_w[wid][k];
        if (a.ids_user) a.ids_user[o] = s_ids[wid][k];
        if (a.w_user) a.w_user[o] = s_w[wid][k];
    }
    if (lane == 0) {
        const float sg = 1.0f / (1.0f + expf(-s_gate[wid]));
        a.sig[t] = sg;
        if (a.sig_user) a.sig_user[t] = sg;
    }
}

// -------------------------------------------------------------- bucketing
// Tokens per counting block: kPfTokBlock * K pairs are counted and scattered
// by one CTA.
constexpr int kPfTokBlock = 32;

__global__ void __launch_bounds__(256) k_pf_count(const int32_t* ids, int T, int K, int E,
                                                  int32_t* cnt_blk) {
    __shared__ int hist[kMaxExperts];
    pdl_launch();
    pdl_wait();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int p0 = blockIdx.x * kPfTokBlock * K;
    const int p1 = min(T * K, p0 + kPfTokBlock * K);
    for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const int e = __ldcg(ids + p);
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cnt_blk[size_t(blockIdx.x) * E + e] = hist[e];
}

// Exclusive scan of one value per thread over the CTA (blockDim <= 1024).
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int r = 0;
        for (int w = 0; w < nw; ++w) {
            const int c = s_warp[w];
            s_warp[w] = r;
            r += c;
        }
        s_warp[32] = r;
    }
    __syncthreads();
    const int ex = s_warp[wid] + incl - v;
    *total = s_warp[32];
    __syncthreads();
    return ex;
}

// The 128-row blocks of every group, largest first, so that the expert
// GEMMs' persistent CTAs, which take the block list's tiles in rounds, end
// their last rounds together: every full block (routed experts ascending,
// then the shared expert), then the partial blocks by descending row count
// (blocks of equal size in any order -- each block's products are its own,
// so the order moves work between CTAs, never a result).  largest_first =
// false keeps expert order (groups of a few tokens, where every block is
// small and the sort's scans cost more than they balance).  Every thread of
// the CTA calls it with the same largest_first; thread e < E brings expert
// e's slots [off, off + total), the others total = 0.  s_bin: kBM + 1 ints.
__device__ void emit_mblocks(int off, int total, int E, int T, bool with_shared,
                             bool largest_first, MBlock* out, int32_t* n_out, int* s_warp,
                             int* s_bin) {
    const int tid = threadIdx.x;
    if (!largest_first) {
        const int nmb = (total + kBM - 1) / kBM, nsh = with_shared ? T : 0;
        int sum_mb = 0;
        const int mbo = block_exclusive_scan(nmb, s_warp, &sum_mb);
        for (int j = 0; j < nmb; ++j)
            out[mbo + j] = MBlock{tid, off + j * kBM, min(kBM, total - j * kBM), 0};
        if (tid == 0) {
            const int nshb = (nsh + kBM - 1) / kBM;
            for (int j = 0; j < nshb; ++j)
                out[sum_mb + j] = MBlock{E, j * kBM, min(kBM, nsh - j * kBM), 0};
            n_out[0] = sum_mb + nshb;
        }
        return;
    }
    for (int i = tid; i <= kBM; i += blockDim.x) s_bin[i] = 0;
    __syncthreads();
    const int nfull = total / kBM, rem = total % kBM;
    const int nsh = with_shared ? T : 0, shfull = nsh / kBM, shrem = nsh % kBM;
    // bin kBM - r holds the partial blocks of r rows: ascending bins are
    // descending sizes
    const int rank = rem > 0 ? atomicAdd(&s_bin[kBM - rem], 1) : 0;
    const int shrank = (tid == 0 && shrem > 0) ? atomicAdd(&s_bin[kBM - shrem], 1) : 0;
    int sum_full = 0;
    const int fo = block_exclusive_scan(nfull, s_warp, &sum_full);
    const int bc = (tid >= 1 && tid < kBM) ? s_bin[tid] : 0;
    int npart = 0;
    const int bstart = block_exclusive_scan(bc, s_warp, &npart);
    if (tid >= 1 && tid < kBM) s_bin[tid] = bstart;
    __syncthreads();
    const int part0 = sum_full + shfull;
    for (int j = 0; j < nfull; ++j) out[fo + j] = MBlock{tid, off + j * kBM, kBM, 0};
    if (rem > 0) out[part0 + s_bin[kBM - rem] + rank] = MBlock{tid, off + nfull * kBM, rem, 0};
    if (tid == 0) {
        for (int j = 0; j < shfull; ++j) out[sum_full + j] = MBlock{E, j * kBM, kBM, 0};
        if (shrem > 0)
            out[part0 + s_bin[kBM - shrem] + shrank] = MBlock{E, shfull * kBM, shrem, 0};
        n_out[0] = part0 + npart;
    }
}

// One CTA of 1024 threads: per-expert totals, offsets, the per-block bases
// of the scatter, and the 128-row blocks of every group (the routed
// experts' and the shared expert's over all T tokens), largest first.
// P threads an expert (P * E <= 1024) each take a contiguous range of the
// counting blocks, so the counts come in one round of loads per pass instead
// of nblk / P; thread e + E p holds part p of expert e (neighbouring threads
// read neighbouring experts' counts).
__global__ void __launch_bounds__(1024) k_pf_scan(PfScanLaunch a) {
    __shared__ int s_warp[33];
    __shared__ int s_bin[kBM + 1];
    __shared__ int s_part[1024];
    pdl_launch();
    pdl_wait();
    const int E = a.E, nb = a.nblk, tid = threadIdx.x;
    const int P = max(1, min(int(blockDim.x) / E, nb));
    const int e = tid % E, part = tid / E;
    const bool act = part < P;
    const int b_lo = act ? int((long long)part * nb / P) : 0;
    const int b_hi = act ? int((long long)(part + 1) * nb / P) : 0;
    constexpr int CH = 16;                // counts loaded CH blocks at a time
    int sum = 0;
    int c1[CH];                           // kept for the second pass when one chunk is all
    for (int b0 = b_lo; b0 < b_hi; b0 += CH) {
        int* c = c1;
#pragma unroll
        for (int j = 0; j < CH; ++j)
            c[j] = (b0 + j < b_hi) ? __ldcg(a.cnt_blk + size_t(b0 + j) * E + e) : 0;
#pragma unroll
        for (int j = 0; j < CH; ++j) sum += c[j];
    }
    s_part[tid] = sum;
    __syncthreads();
    int pre = 0, total = 0;               // the parts before this one; all parts
    if (act)
        for (int p = 0; p < P; ++p) {
            const int v = s_part[p * E + e];
            pre += p < part ? v : 0;
            total += v;
        }
    // thread e < E (part 0) brings expert e to the scans
    const int tot_e = tid < E ? total : 0;
    int sum_slots = 0;
    const int off = block_exclusive_scan(tot_e, s_warp, &sum_slots);
    if (tid < E) {
        a.counts[tid] = tot_e;
        a.offsets[tid] = off;
        s_part[tid] = off;                // every part reads it below
    }
    if (tid == 0) a.offsets[E] = sum_slots;
    __syncthreads();
    if (act) {
        int run = s_part[e] + pre;
        for (int b0 = b_lo; b0 < b_hi; b0 += CH) {
            int c[CH];
#pragma unroll
            for (int j = 0; j < CH; ++j)
                c[j] = (b_hi - b_lo <= CH) ? c1[j]
                       : (b0 + j < b_hi) ? __ldcg(a.cnt_blk + size_t(b0 + j) * E + e) : 0;
#pragma unroll
            for (int j = 0; j < CH; ++j)
                if (b0 + j < b_hi) {
                    a.base_blk[size_t(b0 + j) * E + e] = run;
                    run += c[j];
                }
        }
    }
    emit_mblocks(off, tot_e, E, a.T, a.with_shared != 0, true, a.mblocks, a.n_mblocks, s_warp,
                 s_bin);
}

// The 128-row blocks of the routed slots from caller-supplied offsets (one
// thread an expert; an expert whose range leaves [0, T*K] is skipped and
// latches STRATA_EBADROUTE) and, with_shared, of the shared expert's tokens;
// largest first.
__global__ void __launch_bounds__(1024) k_pf_blocks(const int32_t* offsets, int T, int K, int E,
                                                    int with_shared, MBlock* mblocks,
                                                    int32_t* n_mblocks, uint32_t* err) {
    __shared__ int s_warp[33];
    __shared__ int s_bin[kBM + 1];
    pdl_launch();
    pdl_wait();
    const int e = threadIdx.x;
    int off = 0, total = 0;
    if (offsets != nullptr && e < E) {
        off = __ldg(offsets + e);
        total = __ldg(offsets + e + 1) - off;
        if (off < 0 || total < 0 || (long long)off + total > (long long)T * K) {
            latch(err, STRATA_EBADROUTE);
            total = 0;
        }
    }
    emit_mblocks(off, total, E, T, with_shared != 0, true, mblocks, n_mblocks, s_warp, s_bin);
}

// The three bucketing kernels in one CTA when every pair fits one counting
// block (T <= kPfTokBlock): histogram, offsets and block list, then each
// pair's slot (the expert's offset + its rank among the expert's earlier
// pairs) -- the same slots as k_pf_count / k_pf_scan / k_pf_scatter.
__global__ void __launch_bounds__(1024) k_pf_bucket_small(PfScanLaunch a, const int32_t* ids,
                                                          int K, int32_t* perm, int32_t* inv,
                                                          uint32_t* err) {
    __shared__ int s_ids[kPfTokBlock * kMaxTopK];
    __shared__ int hist[kMaxExperts];
    __shared__ int s_warp[33];
    __shared__ int s_bin[kBM + 1];
    pdl_launch();
    pdl_wait();
    const int E = a.E, TK = a.T * K, tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) hist[e] = 0;
    for (int i = tid; i < TK; i += blockDim.x) s_ids[i] = __ldcg(ids + i);
    __syncthreads();
    for (int i = tid; i < TK; i += blockDim.x) {
        const int e = s_ids[i];
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    const int e = tid;                    // E <= 1024: one expert a thread
    const int total = e < E ? hist[e] : 0;
    int sum_slots = 0;
    const int off = block_exclusive_scan(total, s_warp, &sum_slots);
    if (e < E) {
        a.counts[e] = total;
        a.offsets[e] = off;
        hist[e] = off;                    // from here: the expert's first slot
    }
    if (tid == 0) a.offsets[E] = sum_slots;
    emit_mblocks(off, total, E, a.T, a.with_shared != 0, false, a.mblocks, a.n_mblocks, s_warp,
                 s_bin);
    __syncthreads();
    for (int i = tid; i < TK; i += blockDim.x) {
        const int ei = s_ids[i];
        if (ei < 0 || ei >= E) {
            latch(err, STRATA_EBADROUTE);
            inv[i] = -1;
            continue;
        }
        int rank = 0;
        for (int j = 0; j < i; ++j) rank += (s_ids[j] == ei) ? 1 : 0;
        const int slot = hist[ei] + rank;
        perm[slot] = i;
        inv[i] = slot;
    }
}

// Slots of the block's pairs: base of (block, expert) + rank among the
// block's earlier pairs of the same expert (pairs in ascending t*K + k, so
// an expert's slots ascend in t).
__global__ void __launch_bounds__(256) k_pf_scatter(const int32_t* ids, int T, int K, int E,
                                                    const int32_t* base_blk, int32_t* perm,
                                                    int32_t* inv, uint32_t* err) {
    __shared__ int s_ids[kPfTokBlock * kMaxTopK];
    pdl_launch();
    pdl_wait();
    const int p0 = blockIdx.x * kPfTokBlock * K;
    const int n = min(T * K, p0 + kPfTokBlock * K) - p0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_ids[i] = __ldcg(ids + p0 + i);
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int e = s_ids[i];
        if (e < 0 || e >= E) {
            latch(err, STRATA_EBADROUTE);
            inv[p0 + i] = -1;
            continue;
        }
        int rank = 0;
        for (int j = 0; j < i; ++j) rank += (s_ids[j] == e) ? 1 : 0;
        const int slot = __ldcg(base_blk + size_t(blockIdx.x) * E + e) + rank;
        perm[slot] = p0 + i;
        inv[p0 + i] = slot;
    }
}

// xg[row] = fp16(x[token(row)]) in the operand order; rows < T*K are the
// routed slots (token perm[row] / K), the next T rows the tokens in order.
// A thread takes four 8-element groups of one row, a quarter row apart (so
// neighbouring threads stay on neighbouring groups): one slot lookup, then
// four independent 16-byte loads in flight (H % 32 == 0).
constexpr int kGatherPer = 4;

__global__ void k_pf_gather(const uint16_t* x, const int32_t* perm, int T, int K, int H,
                            __half* xg, int nrows, uint32_t* err) {
    pdl_launch();
    pdl_wait();
    const int gq = H / (8 * kGatherPer);               // groups in a quarter row
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)nrows * gq) return;
    const int row = int(i / gq), g0 = int(i % gq);
    int t;
    if (row < T * K) {
        const int p = __ldcg(perm + row);
        t = (p >= 0 && p < T * K) ? p / K : -1;
    } else {
        t = row - T * K;
    }
    uint4 v[kGatherPer];
#pragma unroll
    for (int q = 0; q < kGatherPer; ++q)
        v[q] = t >= 0 ? __ldg(reinterpret_cast<const uint4*>(x + size_t(t) * H) + g0 + q * gq)
                      : make_uint4(0u, 0u, 0u, 0u);
    uint32_t inf_nan = 0u;       // an fp16 result with an all-ones exponent
#pragma unroll
    for (int q = 0; q < kGatherPer; ++q) {
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (t >= 0) {
            const uint32_t wv[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
            float f[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = bf16_lo(wv[j]);
                f[2 * j + 1] = bf16_hi(wv[j]);
            }
            // positions [0,4,1,5,2,6,3,7]
            const __half2 h0 = __floats2half2_rn(f[0], f[4]);
            const __half2 h1 = __floats2half2_rn(f[1], f[5]);
            const __half2 h2 = __floats2half2_rn(f[2], f[6]);
            const __half2 h3 = __floats2half2_rn(f[3], f[7]);
            out = make_uint4(*reinterpret_cast<const uint32_t*>(&h0),
                             *reinterpret_cast<const uint32_t*>(&h1),
                             *reinterpret_cast<const uint32_t*>(&h2),
                             *reinterpret_cast<const uint32_t*>(&h3));
            const uint32_t bad = bf16x2_over_f16(wv[0]) | bf16x2_over_f16(wv[1]) |
                                 bf16x2_over_f16(wv[2]) | bf16x2_over_f16(wv[3]);
            inf_nan |= bad;
            if (bad != 0u)            // rare: the operand stays finite
                out = make_uint4(f16x2_saturate(out.x), f16x2_saturate(out.y),
                                 f16x2_saturate(out.z), f16x2_saturate(out.w));
        }
        reinterpret_cast<uint4*>(xg + size_t(row) * H)[g0 + q * gq] = out;
    }
    latch_warp(err, STRATA_ERANGE, __ballot_sync(__activemask(), inf_nan != 0u));
}

// fp32 -> fp16 in the operand order, 8 elements a thread.
__global__ void k_pf_pack(const float* src, long long n8, __half* dst, uint32_t* err) {
    pdl_launch();
    pdl_wait();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const float4 a = __ldcg(reinterpret_cast<const float4*>(src) + 2 * i);
    const float4 b = __ldcg(reinterpret_cast<const float4*>(src) + 2 * i + 1);
    const __half2 h0 = __floats2half2_rn(a.x, b.x);
    const __half2 h1 = __floats2half2_rn(a.y, b.y);
    const __half2 h2 = __floats2half2_rn(a.z, b.z);
    const __half2 h3 = __floats2half2_rn(a.w, b.w);
    uint4 out = make_uint4(*reinterpret_cast<const uint32_t*>(&h0),
                           *reinterpret_cast<const uint32_t*>(&h1),
                           *reinterpret_cast<const uint32_t*>(&h2),
                           *reinterpret_cast<const uint32_t*>(&h3));
    const uint32_t bad = f16x2_not_finite(out.x) | f16x2_not_finite(out.y) |
                         f16x2_not_finite(out.z) | f16x2_not_finite(out.w);
    if (bad != 0u)
        out = make_uint4(f16x2_saturate(out.x), f16x2_saturate(out.y), f16x2_saturate(out.z),
                         f16x2_saturate(out.w));
    reinterpret_cast<uint4*>(dst)[i] = out;
    latch_warp(err, STRATA_ERANGE, __ballot_sync(__activemask(), bad != 0u));
}

// out[t] = bf16( sum_k w[t][k] y[inv[t*K+k]] + sig[t] y_sh[t] ), 8 columns
// a thread, k ascending; y in fp16.  resid (optional) += the bf16 output.
__device__ __forceinline__ void h8_to_f32(const uint4& v, float (&f)[8]) {
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&wv[j]));
        f[2 * j] = p.x;
        f[2 * j + 1] = p.y;
    }
}

__device__ __forceinline__ void b8_to_f32(const uint4& v, float (&f)[8]) {
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = bf16_lo(wv[j]);
        f[2 * j + 1] = bf16_hi(wv[j]);
    }
}

template <bool Y_BF16>
__global__ void k_pf_combine(const void* y, const __half* y_sh, const int32_t* inv,
                             const float* w, const float* sig, int T, int K, int H,
                             uint16_t* out, float* resid, uint32_t* err) {
    pdl_launch();
    pdl_wait();
    const int groups = H >> 3;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * groups) return;
    const int t = int(i / groups), g = int(i % groups);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int k = 0; k < K; ++k) {
        const int sl = __ldcg(inv + size_t(t) * K + k);
        if (sl < 0 || sl >= T * K) continue;
        const float wk = __ldcg(w + size_t(t) * K + k);
        float f[8];
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(y) + (size_t(sl) * H + 8 * g) / 8);
        if (Y_BF16)
            b8_to_f32(v, f);
        else
            h8_to_f32(v, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += wk * f[j];
    }
    const float s = __ldcg(sig + t);
    float f[8];
    h8_to_f32(__ldcg(reinterpret_cast<const uint4*>(y_sh + size_t(t) * H + 8 * g)), f);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a0 = acc[2 * j] + s * f[2 * j];
        const float a1 = acc[2 * j + 1] + s * f[2 * j + 1];
        o[j] = uint32_t(f32_to_bf16(a0)) | (uint32_t(f32_to_bf16(a1)) << 16);
    }
    *reinterpret_cast<uint4*>(out + size_t(t) * H + 8 * g) = make_uint4(o[0], o[1], o[2], o[3]);
    // an expert output that overflowed its fp16 copy shows here as a
    // non-finite output (the down products' epilogue carries no check)
    const uint32_t bad = bf16x2_not_finite(o[0]) | bf16x2_not_finite(o[1]) |
                         bf16x2_not_finite(o[2]) | bf16x2_not_finite(o[3]);
    latch_warp(err, STRATA_ERANGE, __ballot_sync(__activemask(), bad != 0u));
    if (resid) {
        float* rr = resid + size_t(t) * H + 8 * g;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            rr[2 * j] += bf16_lo(o[j]);
            rr[2 * j + 1] += bf16_hi(o[j]);
        }
    }
}

// The same sums for few tokens, where the grid is too small to hide
// latency: every pick's slot index and weight, then every pick's row, are
// loaded before any sum (two round trips instead of 2 K).  At many tokens
// the registers this takes cost more occupancy than the loads save.
template <bool Y_BF16, int MAXK>
__global__ void __launch_bounds__(256)
    k_pf_combine_few(const void* y, const __half* y_sh, const int32_t* inv,
                             const float* w, const float* sig, int T, int K, int H,
                             uint16_t* out, float* resid, uint32_t* err) {
    pdl_launch();
    pdl_wait();
    const int groups = H >> 3;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * groups) return;
    const int t = int(i / groups), g = int(i % groups);
    // every slot index and weight, then every slot's row, before any sum:
    // the loads of the K picks are in flight together
    int sl[MAXK];
    float wk[MAXK];
#pragma unroll
    for (int k = 0; k < MAXK; ++k) {
        sl[k] = k < K ? __ldcg(inv + size_t(t) * K + k) : -1;
        wk[k] = k < K ? __ldcg(w + size_t(t) * K + k) : 0.0f;
    }
    uint4 v[MAXK];
#pragma unroll
    for (int k = 0; k < MAXK; ++k) {
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (sl[k] >= 0 && sl[k] < T * K)
            v[k] = __ldcg(reinterpret_cast<const uint4*>(y) + (size_t(sl[k]) * H + 8 * g) / 8);
    }
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < MAXK; ++k) {
        if (sl[k] < 0 || sl[k] >= T * K) continue;          // also k >= K
        float f[8];
        if (Y_BF16)
            b8_to_f32(v[k], f);
        else
            h8_to_f32(v[k], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += wk[k] * f[j];
    }
    const float s = __ldcg(sig + t);
    float f[8];
    h8_to_f32(__ldcg(reinterpret_cast<const uint4*>(y_sh + size_t(t) * H + 8 * g)), f);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a0 = acc[2 * j] + s * f[2 * j];
        const float a1 = acc[2 * j + 1] + s * f[2 * j + 1];
        o[j] = uint32_t(f32_to_bf16(a0)) | (uint32_t(f32_to_bf16(a1)) << 16);
    }
    *reinterpret_cast<uint4*>(out + size_t(t) * H + 8 * g) = make_uint4(o[0], o[1], o[2], o[3]);
    // an expert output that overflowed its fp16 copy shows here as a
    // non-finite output (the down products' epilogue carries no check)
    const uint32_t bad = bf16x2_not_finite(o[0]) | bf16x2_not_finite(o[1]) |
                         bf16x2_not_finite(o[2]) | bf16x2_not_finite(o[3]);
    latch_warp(err, STRATA_ERANGE, __ballot_sync(__activemask(), bad != 0u));
    if (resid) {
        float* rr = resid + size_t(t) * H + 8 * g;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            rr[2 * j] += bf16_lo(o[j]);
            rr[2 * j + 1] += bf16_hi(o[j]);
        }
    }
}

// ------------------------------------------------------------ router GEMM
// K slices of logits^T = router * x^T on the tensor cores.  A = 128 router
// rows (experts; the tile past the last expert holds the shared-gate row and
// the TMA's zero fill), B = 256 tokens, both bf16, K-major, 64-wide K blocks
// by TMA with the 128-byte swizzle; fp32 accumulator in TMEM.  With the
// experts along the TMEM lanes a warp's store writes 32 consecutive logits of
// one token.  One CTA takes one (expert tile, token tile, K slice) and writes
// its partial products; the selection adds the slices in slice order, so the
// result does not depend on scheduling.
constexpr int kRtThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
// Tokens per tile: 256, or 64 for calls of at most 64 tokens (a smaller box
// to fill and MMAs of N = 64 instead of N = 256 over mostly zero rows).
constexpr int kRtBNMax = 256;
constexpr int kRtBNSmall = 64;
constexpr int kRtStages = 4;
constexpr uint32_t kRtABytes = kBM * 128u;
template <int BN>
__host__ __device__ constexpr uint32_t rt_stage_bytes() {
    return kRtABytes + uint32_t(BN) * 128u;
}

struct RouterLaunch {
    float* part;               // [S][T][E + 1]
    const float* bias;         // [E] or NULL: added into slice 0
    uint32_t* err;
    int T, E, S, kbt, n_ttiles;
};

template <int BN>
__global__ void __launch_bounds__(kRtThreads, 1)
    k_pf_router(const __grid_constant__ CUtensorMap map_r, const __grid_constant__ CUtensorMap map_x,
                RouterLaunch a) {
    extern __shared__ uint8_t rt_dyn[];
    __shared__ __align__(8) uint64_t full[kRtStages], empty[kRtStages];
    __shared__ __align__(8) uint64_t acc_full;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rt_dyn) + 1023) &
                                               ~uintptr_t(1023));
    const int item = blockIdx.x;
    const int sl = item % a.S, nt = (item / a.S) % a.n_ttiles, mt = item / (a.S * a.n_ttiles);
    const int kb0 = sl * a.kbt / a.S, nkb = (sl + 1) * a.kbt / a.S - kb0;   // S <= kbt: nkb >= 1

    pdl_launch();
    if (tid == 0) {
        for (int i = 0; i < kRtStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_fence_init();
        tma_prefetch_map(&map_r);
        tma_prefetch_map(&map_x);
    }
    if (wid == 1) {
        tmem_alloc(&tmem_base, BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    const uint32_t tmem = tmem_base;

    if (wid == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kRtStages, round = kb / kRtStages;
                if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1))
                    latch_timeout(a.err, 50, s, round, item);
                uint8_t* st = base + size_t(s) * rt_stage_bytes<BN>();
                mbar_expect_tx(&full[s], rt_stage_bytes<BN>());
                tma_load_2d(st, &map_r, (kb0 + kb) * kBK, mt * kBM, &full[s]);
                tma_load_2d(st + kRtABytes, &map_x, (kb0 + kb) * kBK, nt * BN, &full[s]);
            }
            // every copy has landed before the CTA exits
            for (int i = 0; i < kRtStages && i < nkb; ++i) {
                const int kb = nkb - 1 - i;
                mbar_wait(&full[kb % kRtStages], (kb / kRtStages) & 1);
            }
        }
    } else if (wid == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(kBM, BN, 1);
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kRtStages, round = kb / kRtStages;
                if (!mbar_wait(&full[s], round & 1)) latch_timeout(a.err, 51, s, round, item);
                tc_fence_after();
                const uint32_t st = smem_u32(base + size_t(s) * rt_stage_bytes<BN>());
                const uint64_t ad = sdesc_k_sw128(st), bd = sdesc_k_sw128(st + kRtABytes);
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j)      // + 32 bytes a K step
                    umma_f16(tmem, ad + uint64_t(2 * j), bd + uint64_t(2 * j), idesc,
                             (kb | j) != 0 ? 1u : 0u);
                umma_commit(&empty[s]);
            }
            umma_commit(&acc_full);
            mbar_wait(&acc_full, 0);
        }
    } else {
        // warp w reads TMEM lanes 32 (w % 4) .. +32: router rows (logit columns)
        const int q = wid & 3;
        const int r = mt * kBM + q * 32 + lane;
        const size_t ld = size_t(a.E) + 1;
        float* out = a.part + size_t(sl) * size_t(a.T) * ld + r;
        // slice 0 carries the bias (read while the products run)
        const float b = (sl == 0 && a.bias != nullptr && r < a.E) ? __ldg(a.bias + r) : 0.0f;
        if (!mbar_wait(&acc_full, 0)) latch_timeout(a.err, 52, 0, 0, item);
        tc_fence_after();
        const int t0 = nt * BN;
        for (int c = 0; c < BN / 32 && t0 + 32 * c < a.T; ++c) {    // warp-uniform
            uint32_t v[32];
            tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(32 * c), v);
            tmem_ld_wait();
            if (r <= a.E) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = t0 + 32 * c + j;
                    if (t < a.T) out[size_t(t) * ld] = __uint_as_float(v[j]) + b;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (wid == 1) tmem_dealloc(tmem, BN);
}

// ------------------------------------------------------------------ host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D map over a row-major [rows][inner] array (inner in elements).
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
              uint64_t rows, uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t gdim[2] = {inner, rows};
    const cuuint64_t gstride[1] = {inner * uint64_t(esize)};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r =
        fn(m, dt, 2, const_cast<void*>(base), gdim, gstride, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE,
           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                       Args... args) {
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

}  // namespace

bool prefill_supported(const strata_moe_dims& d) {
    // tile and box rules: K multiples of 256 (two pipeline stages a weight
    // box, >= 16 bytes of scales per row), N multiples of 128, at most 1024
    // experts, and the GEMMs' shared memory at the largest K
    const int kmax = d.hidden > d.inter ? (d.hidden > d.shared_inter ? d.hidden : d.shared_inter)
                                        : (d.inter > d.shared_inter ? d.inter : d.shared_inter);
    return d.inter >= 256 && d.shared_inter >= 256 && d.hidden % 256 == 0 &&
           d.inter % 256 == 0 && d.shared_inter % 256 == 0 && prefill_gemm_fits(kmax);
}

cudaError_t launch_prefill_route(const PfRoute& r, cudaStream_t s) {
    // logit slices: router rows in 128-row boxes, tokens in 256- or 64-row boxes
    CUtensorMap mr, mx;
    if (!make_map(&mr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, r.router, r.H, r.E + 1, kBK, kBM, true) ||
        !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, r.x, r.H, r.T, kBK,
                  r.T <= kRtBNSmall ? kRtBNSmall : kRtBNMax, true))
        return cudaErrorInvalidValue;
    const bool small = r.T <= kRtBNSmall;
    const int BN = small ? kRtBNSmall : kRtBNMax;
    const int n_mt = (r.E + 1 + kBM - 1) / kBM, n_tt = (r.T + BN - 1) / BN, kbt = r.H / kBK;
    // enough K slices to give every SM one tile
    int S = device_info().sms / (n_mt * n_tt);
    S = S < 1 ? 1 : (S > kRouterSplitMax ? kRouterSplitMax : S);
    S = S > kbt ? kbt : S;
    RouterLaunch g{r.part, r.bias, r.err, r.T, r.E, S, kbt, n_tt};
    const size_t dyn =
        size_t(kRtStages) * (small ? rt_stage_bytes<kRtBNSmall>() : rt_stage_bytes<kRtBNMax>()) +
        1024;
    auto go = [&](auto kern) {
        cudaError_t ee =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn));
        return ee != cudaSuccess ? ee
                                 : launch_pdl(kern, n_mt * n_tt * S, kRtThreads, dyn, s, mr, mx, g);
    };
    cudaError_t e = small ? go(k_pf_router<kRtBNSmall>) : go(k_pf_router<kRtBNMax>);
    if (e != cudaSuccess) return e;
    PfSelectLaunch sl{};
    sl.part = r.part;
    sl.nsplit = S;
    sl.logits_user = r.logits_user;
    sl.forced_ids = r.forced_ids;
    sl.forced_w = r.forced_w;
    sl.ids = r.ids;
    sl.w = r.w;
    sl.sig = r.sig;
    sl.ids_user = r.ids_user;
    sl.w_user = r.w_user;
    sl.sig_user = r.sig_user;
    sl.err = r.err;
    sl.T = r.T;
    sl.E = r.E;
    sl.K = r.K;
    const size_t sdyn = size_t(8) * (r.E + 16) * sizeof(float);
    const int grid = (r.T + 7) / 8, nr = (r.E + 1 + 31) / 32;
    if (nr <= 2) return launch_pdl(k_pf_select<2>, grid, 256, sdyn, s, sl);
    if (nr <= 5) return launch_pdl(k_pf_select<5>, grid, 256, sdyn, s, sl);
    if (nr <= 9) return launch_pdl(k_pf_select<9>, grid, 256, sdyn, s, sl);
    return launch_pdl(k_pf_select<0>, grid, 256, sdyn, s, sl);
}

cudaError_t launch_prefill_bucket(const PfBucket& b, cudaStream_t s) {
    const int nblk = (b.T + kPfTokBlock - 1) / kPfTokBlock;
    PfScanLaunch sc{};
    sc.cnt_blk = b.cnt_blk;
    sc.base_blk = b.base_blk;
    sc.counts = b.counts;
    sc.offsets = b.offsets;
    sc.mblocks = b.mblocks;
    sc.n_mblocks = b.n_mblocks;
    sc.nblk = nblk;
    sc.E = b.E;
    sc.T = b.T;
    sc.with_shared = b.with_shared;
    if (nblk == 1)          // every pair in one counting block: one kernel
        return launch_pdl(k_pf_bucket_small, 1, 1024, 0, s, sc, b.ids, b.K, b.perm, b.inv, b.err);
    cudaError_t e = launch_pdl(k_pf_count, nblk, 256, 0, s, b.ids, b.T, b.K, b.E, b.cnt_blk);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_pf_scan, 1, 1024, 0, s, sc);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_pf_scatter, nblk, 256, 0, s, b.ids, b.T, b.K, b.E,
                      static_cast<const int32_t*>(b.base_blk), b.perm, b.inv, b.err);
}

cudaError_t launch_prefill_blocks(const int32_t* offsets, int T, int K, int E, int with_shared,
                                  MBlock* mblocks, int32_t* n_mblocks, uint32_t* err,
                                  cudaStream_t s) {
    return launch_pdl(k_pf_blocks, 1, 1024, 0, s, offsets, T, K, E, with_shared, mblocks,
                      n_mblocks, err);
}

cudaError_t launch_prefill_gather(const uint16_t* x, const int32_t* perm, int T, int K, int H,
                                  __half* xg, int rows, uint32_t* err, cudaStream_t s) {
    if (H % (8 * kGatherPer) != 0) return cudaErrorInvalidValue;
    const long long n = (long long)rows * (H / (8 * kGatherPer));
    return launch_pdl(k_pf_gather, int((n + 255) / 256), 256, 0, s, x, perm, T, K, H, xg, rows,
                      err);
}

cudaError_t launch_prefill_pack(const float* src, long long n, __half* dst, uint32_t* err,
                                cudaStream_t s) {
    const long long n8 = n / 8;
    return launch_pdl(k_pf_pack, int((n8 + 255) / 256), 256, 0, s, src, n8, dst, err);
}

cudaError_t launch_prefill_experts(const PfExperts& p, cudaStream_t s) {
    cudaError_t e = launch_prefill_gather(p.x, p.perm, p.T, p.K, p.H, p.xg, p.xg_rows, p.err, s);
    if (e != cudaSuccess) return e;
    e = launch_prefill_gate_up(p, s);
    if (e != cudaSuccess) return e;
    return launch_prefill_down(p, s);
}

// Below this token count the combine loads every pick before summing.
constexpr int kCombineFewTokens = 256;

cudaError_t launch_prefill_combine(const __half* y_f16, const uint16_t* y_bf16, const __half* ysh,
                                   const int32_t* inv, const float* w, const float* sig, int T,
                                   int K, int H, uint16_t* out, float* resid, uint32_t* err,
                                   cudaStream_t s) {
    const long long n = (long long)T * (H / 8);
    const int grid = int((n + 255) / 256);
    if (T <= kCombineFewTokens && K <= 8) {
        const void* y = y_bf16 != nullptr ? static_cast<const void*>(y_bf16)
                                          : static_cast<const void*>(y_f16);
        if (y_bf16 != nullptr)
            return launch_pdl(k_pf_combine_few<true, 8>, grid, 256, 0, s, y, ysh, inv, w, sig, T,
                              K, H, out, resid, err);
        return launch_pdl(k_pf_combine_few<false, 8>, grid, 256, 0, s, y, ysh, inv, w, sig, T, K,
                          H, out, resid, err);
    }
    if (y_bf16 != nullptr)
        return launch_pdl(k_pf_combine<true>, grid, 256, 0, s, static_cast<const void*>(y_bf16),
                          ysh, inv, w, sig, T, K, H, out, resid, err);
    return launch_pdl(k_pf_combine<false>, grid, 256, 0, s, static_cast<const void*>(y_f16), ysh,
                      inv, w, sig, T, K, H, out, resid, err);
}

}  // namespace strata
