// prefill.cu -- the large-T (prefill) path of the routed MoE FFN on the
// 5th-generation tensor cores.
//
// The pages found the prompt path bound by "dequantize each expert to FP16
// and call oneMKL" (Strata, "Strata on an Intel Arc", section "The engine
// itself on Intel: the SYCL port") and by per-layer host grouping; a fused
// dequant + matrix-unit kernel lost there because it did not overlap the
// two.  Here every step runs on the GPU and the dequantisation feeds the
// tensor cores through shared memory while they run:
//
//   router GEMM     logits = x * router^T (bf16 x bf16 -> fp32, tcgen05)
//   k_pf_select     top-K, softmax weights, sigmoid gate: one warp a token
//   k_pf_count / k_pf_scan / k_pf_scatter
//                   stable counting sort of the (token, k) pairs by expert
//                   and the list of 128-row blocks of every expert ("a
//                   layer's cached experts in a few launches, by how many
//                   rows each has", PolyStrata, "Models and backends",
//                   section "What was tuned"); the shared expert is one more
//                   group whose rows are all tokens
//   k_pf_gather     activations of every slot, fp16, in the operand order
//   gate/up GEMM    persistent tcgen05 kernel: A (activations) by TMA, B =
//                   int4 rows by TMA, dequantised by four warps into the
//                   128-byte-swizzled fp16 tile, fp32 accumulator in TMEM,
//                   SwiGLU in the epilogue -> h (fp16)
//   down GEMM       the same with A = h -> y (bf16)
//   k_pf_combine    out = sum_k w y + sigma(gate) S, in a fixed order
//
// Operand order inside each group of 8 along K: [0,4,1,5,2,6,3,7].  One
// LOP3 on a packed int4 word, (w >> 4j) & 0x000F000F | 0x64006400, yields
// the fp16 pair (1024 + u_j, 1024 + u_{j+4}); writing the activations (A)
// in the same order makes the products the natural ones, since the MMA sums
// over K in any consistent order.

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace strata {

// ------------------------------------------------------------- selection
// One warp a token: top-K (ties to the lower id), ids ascending,
// renormalised softmax weights, sigmoid of the shared-gate logit; or the
// forced ids/weights.  The same arithmetic as the decode path.
__global__ void __launch_bounds__(256) k_pf_select(PfSelectLaunch a) {
    extern __shared__ float s_dyn[];
    pdl_launch();
    pdl_wait();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int t = blockIdx.x * (blockDim.x >> 5) + wid;
    if (t >= a.T) return;
    const int E = a.E, K = a.K;
    const float* lg = a.logits + size_t(t) * (E + 1);
    float* L = s_dyn + size_t(wid) * (E + 16);
    __shared__ int s_ids[8][kMaxTopK];
    __shared__ float s_w[8][kMaxTopK];
    if (a.forced_ids) {
        for (int k = lane; k < K; k += 32) {
            const int id = __ldg(a.forced_ids + size_t(t) * K + k);
            if (id < 0 || id >= E) latch(a.err, STRATA_EBADROUTE);
            s_ids[wid][k] = id;
            s_w[wid][k] = __ldg(a.forced_w + size_t(t) * K + k);
        }
        __syncwarp();
    } else {
        // top-K of the E logits, as in the decode path
        for (int e = lane; e < E; e += 32) L[e] = __ldcg(lg + e);
        __syncwarp();
        float bv = -INFINITY;
        int be = 0x7fffffff;
        for (int e = lane; e < E; e += 32) {
            const float v = L[e];
            if (v > bv || (v == bv && e < be)) {
                bv = v;
                be = e;
            }
        }
        float myv = 0.0f;
        int mye = 0x7fffffff;
        for (int k = 0; k < K; ++k) {
            float wv = bv;
            int we = be;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, we, o);
                if (ov > wv || (ov == wv && oe < we)) {
                    wv = ov;
                    we = oe;
                }
            }
            if (lane == k) {
                myv = wv;
                mye = we;
            }
            if (we < E && (we & 31) == lane) {
                L[we] = __int_as_float(0x7fc00000);
                bv = -INFINITY;
                be = 0x7fffffff;
                for (int e = lane; e < E; e += 32) {
                    const float v = L[e];
                    if (v > bv || (v == bv && e < be)) {
                        bv = v;
                        be = e;
                    }
                }
            }
        }
        const float m = __shfl_sync(0xffffffffu, myv, 0);
        int rank = 0;
        for (int j = 0; j < K; ++j) rank += (__shfl_sync(0xffffffffu, mye, j) < mye) ? 1 : 0;
        float* ex = L + E;
        float e_k = 0.0f;
        if (lane < K) {
            e_k = expf(myv - m);
            ex[rank] = e_k;
            s_ids[wid][rank] = mye;
        }
        __syncwarp();
        float sum = 0.0f;
        for (int r = 0; r < K; ++r) sum += ex[r];
        if (lane < K) s_w[wid][rank] = e_k / sum;
        __syncwarp();
    }
    if (a.logits_user)
        for (int e = lane; e < E; e += 32) a.logits_user[size_t(t) * E + e] = __ldcg(lg + e);
    for (int k = lane; k < K; k += 32) {
        const size_t o = size_t(t) * K + k;
        a.ids[o] = s_ids[wid][k];
        a.w[o] = s_w[wid][k];
        if (a.ids_user) a.ids_user[o] = s_ids[wid][k];
        if (a.w_user) a.w_user[o] = s_w[wid][k];
    }
    if (lane == 0) {
        const float s = 1.0f / (1.0f + expf(-__ldcg(lg + E)));
        a.sig[t] = s;
        if (a.sig_user) a.sig_user[t] = s;
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

// One CTA of 1024 threads: per-expert totals, offsets, the per-block bases
// of the scatter, and the 128-row blocks of every group (routed experts in
// ascending id, then the shared expert over all T tokens).
__global__ void __launch_bounds__(1024) k_pf_scan(PfScanLaunch a) {
    __shared__ int s_warp[33];
    pdl_launch();
    pdl_wait();
    const int E = a.E, nb = a.nblk;
    const int e = threadIdx.x;            // E <= 1024: one expert a thread
    constexpr int CH = 16;                // counts loaded CH blocks at a time
    int total = 0;
    if (e < E) {
        for (int b0 = 0; b0 < nb; b0 += CH) {
            int c[CH];
#pragma unroll
            for (int j = 0; j < CH; ++j)
                c[j] = (b0 + j < nb) ? __ldcg(a.cnt_blk + size_t(b0 + j) * E + e) : 0;
#pragma unroll
            for (int j = 0; j < CH; ++j) total += c[j];
        }
    }
    const int nmb = (total + kBM - 1) / kBM;
    int sum_slots = 0, sum_mb = 0;
    const int off = block_exclusive_scan(total, s_warp, &sum_slots);
    const int mbo = block_exclusive_scan(nmb, s_warp, &sum_mb);
    if (e < E) {
        a.counts[e] = total;
        a.offsets[e] = off;
        int run = off;
        for (int b0 = 0; b0 < nb; b0 += CH) {
            int c[CH];
#pragma unroll
            for (int j = 0; j < CH; ++j)
                c[j] = (b0 + j < nb) ? __ldcg(a.cnt_blk + size_t(b0 + j) * E + e) : 0;
#pragma unroll
            for (int j = 0; j < CH; ++j)
                if (b0 + j < nb) {
                    a.base_blk[size_t(b0 + j) * E + e] = run;
                    run += c[j];
                }
        }
        for (int j = 0; j < nmb; ++j) {
            MBlock mb;
            mb.group = e;
            mb.row = off + j * kBM;
            mb.nrows = min(kBM, total - j * kBM);
            mb.pad = 0;
            a.mblocks[mbo + j] = mb;
        }
    }
    if (threadIdx.x == 0) {
        a.offsets[E] = sum_slots;
        const int nsh = a.with_shared ? (a.T + kBM - 1) / kBM : 0;
        for (int j = 0; j < nsh; ++j) {
            MBlock mb;
            mb.group = E;
            mb.row = j * kBM;
            mb.nrows = min(kBM, a.T - j * kBM);
            mb.pad = 0;
            a.mblocks[sum_mb + j] = mb;
        }
        a.n_mblocks[0] = sum_mb + nsh;
    }
}

// The 128-row blocks of the routed slots from caller-supplied offsets (one
// thread an expert; an expert whose range leaves [0, T*K] is skipped and
// latches STRATA_EBADROUTE) and, with_shared, of the shared expert's tokens.
__global__ void __launch_bounds__(1024) k_pf_blocks(const int32_t* offsets, int T, int K, int E,
                                                    int with_shared, MBlock* mblocks,
                                                    int32_t* n_mblocks, uint32_t* err) {
    __shared__ int s_warp[33];
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
    const int nmb = (total + kBM - 1) / kBM;
    int sum_mb = 0;
    const int mbo = block_exclusive_scan(nmb, s_warp, &sum_mb);
    for (int j = 0; j < nmb; ++j) {
        MBlock mb;
        mb.group = e;
        mb.row = off + j * kBM;
        mb.nrows = min(kBM, total - j * kBM);
        mb.pad = 0;
        mblocks[mbo + j] = mb;
    }
    if (threadIdx.x == 0) {
        const int nsh = with_shared ? (T + kBM - 1) / kBM : 0;
        for (int j = 0; j < nsh; ++j) {
            MBlock mb;
            mb.group = E;
            mb.row = j * kBM;
            mb.nrows = min(kBM, T - j * kBM);
            mb.pad = 0;
            mblocks[sum_mb + j] = mb;
        }
        n_mblocks[0] = sum_mb + nsh;
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
__global__ void k_pf_gather(const uint16_t* x, const int32_t* perm, int T, int K, int H,
                            __half* xg, int nrows) {
    pdl_launch();
    pdl_wait();
    const int groups = H >> 3;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)nrows * groups) return;
    const int row = int(i / groups), g = int(i % groups);
    int t;
    if (row < T * K) {
        const int p = __ldcg(perm + row);
        t = (p >= 0 && p < T * K) ? p / K : -1;
    } else {
        t = row - T * K;
    }
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (t >= 0) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + size_t(t) * H + 8 * g));
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
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
    }
    *reinterpret_cast<uint4*>(xg + size_t(row) * H + 8 * g) = out;
}

// fp32 -> fp16 in the operand order, 8 elements a thread.
__global__ void k_pf_pack(const float* src, long long n8, __half* dst) {
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
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(*reinterpret_cast<const uint32_t*>(&h0),
                                                  *reinterpret_cast<const uint32_t*>(&h1),
                                                  *reinterpret_cast<const uint32_t*>(&h2),
                                                  *reinterpret_cast<const uint32_t*>(&h3));
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
                             uint16_t* out, float* resid) {
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
    if (resid) {
        float* rr = resid + size_t(t) * H + 8 * g;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            rr[2 * j] += bf16_lo(o[j]);
            rr[2 * j + 1] += bf16_hi(o[j]);
        }
    }
}

// ------------------------------------------------------------------ GEMM
// Persistent grouped GEMM, one CTA per SM, six warps:
//   warp 0      TMA producer (A and B stages; the tile's scales)
//   warp 1      TMEM allocation; lane 0 issues the MMAs
//   warps 2..5  dequantise B into the swizzled fp16 tile, then read the
//               accumulator out of TMEM (warp w owns TMEM lanes
//               32 (w % 4) .. +32) and store the tile
// A tile: 128 rows x 64 K (fp16 or bf16), B tile: BN rows x 64 K; the MMA is
// M = 128, N = BN, K = 16, four per stage.
constexpr int kPfThreads = 192;
constexpr int kTmemCols = 256;

struct GemmSmem {
    uint32_t stage_bytes, a_off, b_off, pk_off, sc_off, total;
};

__host__ __device__ inline GemmSmem gemm_smem(int mode, int BN, int K, int stages) {
    GemmSmem s{};
    s.a_off = 0;
    s.b_off = kBM * 128;
    s.pk_off = s.b_off + uint32_t(BN) * 128;
    s.stage_bytes = s.pk_off + (mode == kGemmRouter ? 0u : uint32_t(BN) * 32u);
    s.sc_off = uint32_t(stages) * s.stage_bytes;
    s.total = s.sc_off + (mode == kGemmRouter ? 0u : uint32_t(BN) * uint32_t(K / 32) * 2u);
    return s;
}

// Dequantise one 64-wide K slice of one B row: 32 packed bytes and two
// scales -> 64 fp16 in the operand order, 8 chunks of 16 bytes stored with
// the 128-byte swizzle (chunk c of row r at (c ^ (r & 7)) * 16).
__device__ __forceinline__ void dequant_row64(const uint8_t* pk, const uint16_t* sc2,
                                              uint8_t* brow, int r) {
    const uint4 w0 = *reinterpret_cast<const uint4*>(pk);
    const uint4 w1 = *reinterpret_cast<const uint4*>(pk + 16);
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const __half2 s0 = __halves2half2(__ushort_as_half(sc2[0]), __ushort_as_half(sc2[0]));
    const __half2 s1 = __halves2half2(__ushort_as_half(sc2[1]), __ushort_as_half(sc2[1]));
    const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const __half2 s = (c < 4) ? s0 : s1;
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t b = ((words[c] >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
            const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&b), off);  // exact
            const __half2 v = __hmul2(q, s);
            o[j] = *reinterpret_cast<const uint32_t*>(&v);
        }
        *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kPfThreads, 1)
    k_pf_gemm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_a2,
              const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_bs,
              const __grid_constant__ CUtensorMap map_b2, const __grid_constant__ CUtensorMap map_bs2,
              GemmLaunch a) {
    extern __shared__ uint8_t pf_dyn[];
    __shared__ __align__(8) uint64_t full[kPfMaxStages], deq[kPfMaxStages], empty[kPfMaxStages];
    __shared__ __align__(8) uint64_t acc_full, acc_empty, sc_full, sc_empty;
    __shared__ uint32_t tmem_base;
    __shared__ int s_ntiles;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int S = a.stages, BN = a.BN;
    const bool int4b = MODE != kGemmRouter;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pf_dyn) + 1023) &
                                               ~uintptr_t(1023));
    const GemmSmem L = gemm_smem(MODE, BN, a.K_max, S);

    pdl_launch();
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&deq[i], 128);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, 128);
        mbar_init(&sc_full, 1);
        mbar_init(&sc_empty, 128);
        mbar_fence_init();
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
    }
    if (wid == 1) {
        tmem_alloc(&tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    if (tid == 0) s_ntiles = (MODE == kGemmRouter ? a.router_mblocks : __ldcg(a.n_mblocks)) * a.nb_max;
    __syncthreads();
    const int n_tiles = s_ntiles;
    const uint32_t tmem = tmem_base;
    const uint32_t idesc_full = idesc_f16(kBM, BN, MODE == kGemmRouter ? 1 : 0);

    // tile -> (m-block, n-block); returns false when the n-block does not
    // exist for the m-block's group
    auto tile_info = [&](int tile, int& group, int& row, int& nrows, int& n0, int& N, int& K) {
        const int mb = tile / a.nb_max, nb = tile % a.nb_max;
        if (MODE == kGemmRouter) {
            group = 0;
            row = mb * kBM;
            nrows = min(kBM, a.M - row);
            N = a.N;
            K = a.K;
        } else {
            const MBlock m = a.mblocks[mb];
            group = m.group;
            row = m.row;
            nrows = m.nrows;
            const bool sh = group == a.E;
            N = sh ? a.N2 : a.N;
            K = sh ? a.K2 : a.K;
        }
        n0 = nb * BN;
        return n0 < N;
    };

    if (wid == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kbt = 0, ti = 0;
            for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
                int g, row, nrows, n0, N, K;
                if (!tile_info(tile, g, row, nrows, n0, N, K)) continue;
                const bool sh = int4b && g == a.E;
                const CUtensorMap* ma = (sh && MODE == kGemmDown) ? &map_a2 : &map_a;
                const CUtensorMap* mbq = sh ? &map_b2 : &map_b;
                const CUtensorMap* mbs = sh ? &map_bs2 : &map_bs;
                const int arow = (sh && MODE == kGemmGateUp) ? a.a_shared_row0 + row : row;
                const int brow = (int4b && !sh) ? g * N + n0 : n0;
                if (int4b) {
                    if (ti > 0 && !mbar_wait(&sc_empty, (ti - 1) & 1))
                        latch_timeout(a.err, 11, 0, ti, tile);
                    mbar_expect_tx(&sc_full, uint32_t(BN) * uint32_t(K / 32) * 2u);
                    tma_load_2d(base + L.sc_off, mbs, 0, brow, &sc_full);
                }
                const int kbn = K / kBK;
                for (int kb = 0; kb < kbn; ++kb, ++kbt) {
                    const int s = int(kbt % S);
                    const uint32_t round = kbt / S;
                    if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1))
                        latch_timeout(a.err, 12, s, round, tile);
                    uint8_t* st = base + size_t(s) * L.stage_bytes;
                    const uint32_t bbytes = int4b ? uint32_t(BN) * 32u : uint32_t(BN) * 128u;
                    mbar_expect_tx(&full[s], uint32_t(kBM) * 128u + bbytes);
                    tma_load_2d(st + L.a_off, ma, kb * kBK, arow, &full[s]);
                    if (int4b)
                        tma_load_2d(st + L.pk_off, mbq, kb * (kBK / 2), brow, &full[s]);
                    else
                        tma_load_2d(st + L.b_off, mbq, kb * kBK, brow, &full[s]);
                }
                ++ti;
            }
        }
    } else if (wid == 1) {
        // ----------------------------------------------------------- MMA
        if (lane == 0) {
            uint32_t kbt = 0, ti = 0;
            for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
                int g, row, nrows, n0, N, K;
                if (!tile_info(tile, g, row, nrows, n0, N, K)) continue;
                if (ti > 0 && !mbar_wait(&acc_empty, (ti - 1) & 1))
                    latch_timeout(a.err, 13, 0, ti, tile);
                tc_fence_after();
                const int kbn = K / kBK;
                for (int kb = 0; kb < kbn; ++kb, ++kbt) {
                    const int s = int(kbt % S);
                    const uint32_t round = kbt / S;
                    if (!mbar_wait(int4b ? &deq[s] : &full[s], round & 1))
                        latch_timeout(a.err, 14, s, round, tile);
                    tc_fence_after();
                    const uint32_t st = smem_u32(base + size_t(s) * L.stage_bytes);
#pragma unroll
                    for (int j = 0; j < kBK / 16; ++j) {
                        const uint64_t ad = sdesc_k_sw128(st + L.a_off + 32u * j);
                        const uint64_t bd = sdesc_k_sw128(st + L.b_off + 32u * j);
                        umma_f16(tmem, ad, bd, idesc_full, (kb | j) != 0 ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);
                }
                umma_commit(&acc_full);
                ++ti;
            }
        }
    } else {
        // ---------------------------------------- dequant + epilogue
        const int dq = tid - 64;                 // 0..127
        const int q = wid & 3;                   // TMEM lane quarter of this warp
        const int m = q * 32 + lane;             // accumulator row of this thread
        uint32_t kbt = 0, ti = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            int g, row, nrows, n0, N, K;
            if (!tile_info(tile, g, row, nrows, n0, N, K)) continue;
            const bool sh = int4b && g == a.E;
            const int kbn = K / kBK;
            if (int4b && !mbar_wait(&sc_full, ti & 1)) latch_timeout(a.err, 15, 0, ti, tile);
            const uint16_t* sct = reinterpret_cast<const uint16_t*>(base + L.sc_off);
            for (int kb = 0; kb < kbn; ++kb, ++kbt) {
                const int s = int(kbt % S);
                const uint32_t round = kbt / S;
                if (int4b) {
                    if (!mbar_wait(&full[s], round & 1)) latch_timeout(a.err, 16, s, round, tile);
                    uint8_t* st = base + size_t(s) * L.stage_bytes;
                    for (int r = dq; r < BN; r += 128)
                        dequant_row64(st + L.pk_off + r * 32, sct + size_t(r) * (K / 32) + 2 * kb,
                                      st + L.b_off + r * 128, r);
                    fence_proxy_async_smem();
                    mbar_arrive(&deq[s]);
                }
            }
            if (int4b) mbar_arrive(&sc_empty);

            // epilogue
            if (!mbar_wait(&acc_full, ti & 1)) latch_timeout(a.err, 17, 0, ti, tile);
            tc_fence_after();
            const bool valid = m < nrows;
            const uint32_t tl = tmem + (uint32_t(q * 32) << 16);
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tl + uint32_t(c * 32), v);
                tmem_ld_wait();
                if (!valid) continue;
                const int col0 = n0 + c * 32;
                if (MODE == kGemmRouter) {
                    float* o = a.out_f32 + size_t(row + m) * a.ldo;
                    for (int j = 0; j < 32; ++j) {
                        const int n = col0 + j;
                        if (n < a.N_valid)
                            o[n] = __uint_as_float(v[j]) +
                                   ((a.bias != nullptr && n < a.E) ? __ldg(a.bias + n) : 0.0f);
                    }
                } else if (MODE == kGemmGateUp) {
                    // h_i = silu(gate) * up for 16 pairs, stored in the operand order
                    float hv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        hv[i] = silu_mul(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    const int ld = sh ? a.ld2 : a.ldo;
                    if (!sh && a.out_f32 != nullptr) {
                        // natural order, fp32 (the h of the stage-wise calls)
                        float4* h32 = reinterpret_cast<float4*>(a.out_f32 + size_t(row + m) * ld +
                                                                col0 / 2);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            h32[j] = make_float4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2],
                                                 hv[4 * j + 3]);
                    }
                    __half* hrow = (sh ? a.out2_f16 : a.out_f16) + size_t(row + m) * ld + col0 / 2;
#pragma unroll
                    for (int gq = 0; gq < 2; ++gq) {
                        const float* f = hv + 8 * gq;
                        const __half2 h0 = __floats2half2_rn(f[0], f[4]);
                        const __half2 h1 = __floats2half2_rn(f[1], f[5]);
                        const __half2 h2 = __floats2half2_rn(f[2], f[6]);
                        const __half2 h3 = __floats2half2_rn(f[3], f[7]);
                        *reinterpret_cast<uint4*>(hrow + 8 * gq) =
                            make_uint4(*reinterpret_cast<const uint32_t*>(&h0),
                                       *reinterpret_cast<const uint32_t*>(&h1),
                                       *reinterpret_cast<const uint32_t*>(&h2),
                                       *reinterpret_cast<const uint32_t*>(&h3));
                    }
                } else if (!sh && a.out_bf16 != nullptr) {
                    // y in bf16 (the stage-wise calls' format)
                    uint16_t* yrow = a.out_bf16 + size_t(row + m) * a.ldo + col0;
#pragma unroll
                    for (int gq = 0; gq < 4; ++gq) {
                        uint32_t o[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            o[j] = uint32_t(f32_to_bf16(__uint_as_float(v[8 * gq + 2 * j]))) |
                                   (uint32_t(f32_to_bf16(__uint_as_float(v[8 * gq + 2 * j + 1])))
                                    << 16);
                        *reinterpret_cast<uint4*>(yrow + 8 * gq) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                } else {
                    // y in fp16: the combine sums several of them before the
                    // output's own rounding
                    __half* yrow = (sh ? a.out2_f16 : a.out_f16) + size_t(row + m) * a.ldo + col0;
#pragma unroll
                    for (int gq = 0; gq < 4; ++gq) {
                        uint32_t o[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const __half2 hv2 = __floats2half2_rn(__uint_as_float(v[8 * gq + 2 * j]),
                                                                  __uint_as_float(v[8 * gq + 2 * j + 1]));
                            o[j] = *reinterpret_cast<const uint32_t*>(&hv2);
                        }
                        *reinterpret_cast<uint4*>(yrow + 8 * gq) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty);
            ++ti;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (wid == 1) tmem_dealloc(tmem, kTmemCols);
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

int pick_stages(int mode, int BN, int K) {
    for (int S = kPfMaxStages; S >= 2; --S) {
        const GemmSmem L = gemm_smem(mode, BN, K, S);
        if (L.total + 1024 <= kPfSmemBudget) return S;
    }
    return 0;
}

template <int MODE>
cudaError_t run_gemm(GemmLaunch g, const CUtensorMap& ma, const CUtensorMap& ma2,
                     const CUtensorMap& mb, const CUtensorMap& mbs, const CUtensorMap& mb2,
                     const CUtensorMap& mbs2, cudaStream_t s) {
    const Dev d = device_info();
    g.stages = pick_stages(MODE, g.BN, g.K_max);
    if (g.stages < 2) return cudaErrorInvalidValue;
    const size_t dyn = gemm_smem(MODE, g.BN, g.K_max, g.stages).total + 1024;
    cudaError_t e = cudaFuncSetAttribute(k_pf_gemm<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn));
    if (e != cudaSuccess) return e;
    return launch_pdl(k_pf_gemm<MODE>, d.sms, kPfThreads, dyn, s, ma, ma2, mb, mbs, mb2, mbs2, g);
}

}  // namespace

bool prefill_supported(const strata_moe_dims& d) {
    // tile and box rules: K multiples of 64 with >= 16 bytes of scales per
    // row (K >= 256), N multiples of 128, and at most 1024 experts
    return d.inter >= 256 && d.shared_inter >= 256 && d.hidden % 256 == 0;
}

cudaError_t launch_prefill_route(const PfRoute& r, cudaStream_t s) {
    // logits = x * router^T
    CUtensorMap ma, mb;
    if (!make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, r.x, r.H, r.T, kBK, kBM, true) ||
        !make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, r.router, r.H, r.E + 1, kBK, 128, true))
        return cudaErrorInvalidValue;
    GemmLaunch g{};
    g.BN = 128;
    g.N = r.E + 1;
    g.N_valid = r.E + 1;
    g.K = r.H;
    g.K_max = r.H;
    g.M = r.T;
    g.router_mblocks = (r.T + kBM - 1) / kBM;
    g.nb_max = (r.E + 1 + 127) / 128;
    g.out_f32 = r.logits;
    g.bias = r.bias;
    g.E = r.E;
    g.ldo = r.E + 1;
    g.err = r.err;
    cudaError_t e = run_gemm<kGemmRouter>(g, ma, ma, mb, mb, mb, mb, s);
    if (e != cudaSuccess) return e;
    PfSelectLaunch sl{};
    sl.logits = r.logits;
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
    const size_t dyn = size_t(8) * (r.E + 16) * sizeof(float);
    return launch_pdl(k_pf_select, (r.T + 7) / 8, 256, dyn, s, sl);
}

cudaError_t launch_prefill_bucket(const PfBucket& b, cudaStream_t s) {
    const int nblk = (b.T + kPfTokBlock - 1) / kPfTokBlock;
    cudaError_t e = launch_pdl(k_pf_count, nblk, 256, 0, s, b.ids, b.T, b.K, b.E, b.cnt_blk);
    if (e != cudaSuccess) return e;
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
                                  __half* xg, int rows, cudaStream_t s) {
    const long long n = (long long)rows * (H / 8);
    return launch_pdl(k_pf_gather, int((n + 255) / 256), 256, 0, s, x, perm, T, K, H, xg, rows);
}

cudaError_t launch_prefill_pack(const float* src, long long n, __half* dst, cudaStream_t s) {
    const long long n8 = n / 8;
    return launch_pdl(k_pf_pack, int((n8 + 255) / 256), 256, 0, s, src, n8, dst);
}

cudaError_t launch_prefill_experts(const PfExperts& p, cudaStream_t s) {
    cudaError_t e = launch_prefill_gather(p.x, p.perm, p.T, p.K, p.H, p.xg, p.xg_rows, s);
    if (e != cudaSuccess) return e;
    e = launch_prefill_gate_up(p, s);
    if (e != cudaSuccess) return e;
    return launch_prefill_down(p, s);
}

cudaError_t launch_prefill_combine(const __half* y_f16, const uint16_t* y_bf16, const __half* ysh,
                                   const int32_t* inv, const float* w, const float* sig, int T,
                                   int K, int H, uint16_t* out, float* resid, cudaStream_t s) {
    const long long n = (long long)T * (H / 8);
    const int grid = int((n + 255) / 256);
    if (y_bf16 != nullptr)
        return launch_pdl(k_pf_combine<true>, grid, 256, 0, s, static_cast<const void*>(y_bf16),
                          ysh, inv, w, sig, T, K, H, out, resid);
    return launch_pdl(k_pf_combine<false>, grid, 256, 0, s, static_cast<const void*>(y_f16), ysh,
                      inv, w, sig, T, K, H, out, resid);
}

}  // namespace strata
