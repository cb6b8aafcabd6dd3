// prefill_gemm.cu -- the prefill experts' grouped GEMMs with the weights as
// the tensor cores' A operand in tensor memory (swap AB).
//
// Each tile is 128 weight rows (of one expert, or of the shared expert) by
// the n <= 128 token rows of one block of that expert, over the full K:
//   D[w][t] = sum_k W[w][k] X[t][k]         (fp32 in TMEM, 128 lanes x n cols)
// The int4 weights are dequantised by four warps straight from the packed
// bytes into registers and stored into tensor memory with tcgen05.st, where
// the MMA reads them as its A operand: no dequantised tile goes through
// shared memory, and N follows the expert's token count (rounded up to 16)
// instead of padding every expert to 128 rows.  The activations (B) come by
// TMA into 128-byte-swizzled shared memory, one 3-D box a pipeline stage:
// the block's rows rounded up to 32 (one tensor map per height) by the
// stage's four 64-wide K blocks.
//
// Warps: 0 TMA producer; 1 and 2 the MMAs (lane 0; warp 1 also allocates
// the TMEM); 3..10 dequantisation, two sets of four taking alternate
// stages (warp w owns TMEM lanes 32 (w % 4) .. +32: weight rows); 11..14
// epilogue (the same lane quarters): SwiGLU of gate/up row pairs (rows 2i,
// 2i+1 sit in neighbouring lanes) or the down product's outputs.
// One thread issues a tcgen05.mma about every 54 cycles however small N is,
// while the tensor pipe needs only N / 2 cycles for a 128 x N x 16 product:
// a tile of at most 64 tokens therefore splits its K steps between the two
// MMA warps, each into an accumulator of its own, which the epilogue adds.
// Accumulators are double-buffered (2 x 128 columns) so a tile's epilogue
// overlaps the next tile's MMAs; the dequantised A stages take 2 x 128
// columns.  A pipeline stage is K = 256 (sixteen MMAs): an MMA warp pays
// about 220 cycles a stage for its fence and commit and 70-95 an MMA, so
// fewer, longer stages leave more of its time to the MMAs (K = 128 stages:
// gate/up 158 us, down 94 us at T = 2048; K = 256: 141 and 86).
//
// The pages found a fused dequantise + matrix-unit kernel losing to
// dequantise-then-library-GEMM when the two did not overlap (Strata, "Strata
// on an Intel Arc", section "The engine itself on Intel: the SYCL port");
// here the dequantisation of stage k + 1 runs while the MMA eats stage k.

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace strata {

constexpr int kSabThreads = 480;
constexpr int kSabMmaWarps = 2;          // MMA issuing warps (1, 2)
constexpr int kSabDeq0 = 1 + kSabMmaWarps;   // first dequantisation warp
constexpr int kSabDeqSets = 2;           // dequantisation warp sets: K blocks alternate
constexpr int kSabKS = 256;              // K of one pipeline stage: 16 MMAs of K = 16
constexpr int kSabStages = 2;            // activation stages = dequantised A stages
constexpr int kSabACols = kSabKS / 2;    // TMEM columns of one A stage (two fp16 a column)
constexpr int kSabDCols = 128;           // one accumulator buffer: up to 128 token columns
constexpr int kSabACol0 = 2 * kSabDCols; // first A column
constexpr int kSabTmemCols = 512;
constexpr int kSabBoxRows = 32;          // activation box heights: 32, 64, 96, 128 rows
constexpr int kSabXMaps = kBM / kSabBoxRows;
constexpr uint32_t kSabSubBytes = kBM * 128u;          // 128 rows x 64 fp16 (one MMA K block)
constexpr uint32_t kSabStageBytes = (kSabKS / 64) * kSabSubBytes;  // 64-wide K sub-blocks

// Activation maps of one operand, one per box height (rows 32 (i + 1)).
// The box of map i lands as [4 K blocks][32 (i + 1) rows][64 fp16].
struct SabXMaps {
    CUtensorMap m[kSabXMaps];
};
// Weight stages: 128 rows x 128 packed bytes = 256 inputs = one pipeline
// stage, one TMA box with the 128-byte swizzle, so every row is read from
// memory as a whole 128-byte line and a lane's 16-byte reads of its row are
// spread over the banks.
constexpr uint32_t kSabWRowBytes = 128;  // packed bytes of a row in a weight stage
constexpr uint32_t kSabWBytes = kBM * kSabWRowBytes;
constexpr int kSabWStages = 3;
static_assert(kSabStages * kSabACols + kSabACol0 <= kSabTmemCols, "TMEM columns");
static_assert(kSabKS / 2 == int(kSabWRowBytes), "one weight stage a pipeline stage");

// A tile's scales land as [K / 256][128 rows][8 fp16]: the 8 scales of a
// row for 256 inputs (one pipeline stage) side by side, so a stage's read
// of 16 bytes per row by 32 consecutive rows spans only a few wavefronts
// (row-major [128][K / 32] put all 32 rows of a warp in one bank).
__host__ __device__ inline uint32_t sab_scale_bytes(int K_max) {
    return uint32_t(kBM) * uint32_t(K_max / 32) * 2u;
}

// Dynamic shared memory of the expert GEMM: activation stages, weight
// stages, two scale buffers and the 1024-byte alignment slack.
inline size_t sab_smem_bytes(int K_max) {
    return size_t(kSabStages) * kSabStageBytes + size_t(kSabWStages) * kSabWBytes +
           2 * size_t(sab_scale_bytes(K_max)) + 1024;
}

// 64 fp16 weights of one row for one K block: 32 packed bytes, two scales
// -> 32 registers holding the MMA-order pairs, register c = K positions
// (2c, 2c+1).  Within every 8 elements the positions hold elements
// [0,4,1,5,2,6,3,7], so a pair is one nibble position of the word's two
// 16-bit halves (the activations are stored in the same order, so the
// products are the natural ones).  A nibble n is or-ed into the mantissa of
// 1024.0: at bits 0-3 that reads 1024 + n and a subtraction of 1032 gives
// n - 8; at bits 4-7 it reads 1024 + 16 n and a fused multiply-add with 1/16
// and -72 gives n - 8; both exact.  One shift by 8 brings the upper byte's
// nibbles down, so a word of four pairs costs one shift and four masks on the
// integer pipe, the rest is half2 arithmetic.  The product with the scale is
// the single rounding.
__device__ __forceinline__ void dequant_row_regs(const uint4& w0, const uint4& w1, uint32_t sc2,
                                                 uint32_t (&r)[32]) {
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2c00), __ushort_as_half(0x2c00));
    const __half2 m72 = __halves2half2(__ushort_as_half(0xd480), __ushort_as_half(0xd480));
    const __half s0 = __ushort_as_half(uint16_t(sc2 & 0xffffu));
    const __half s1 = __ushort_as_half(uint16_t(sc2 >> 16));
    const __half2 sA = __halves2half2(s0, s0), sB = __halves2half2(s1, s1);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const __half2 s = (c < 4) ? sA : sB;
        const uint32_t w = words[c], wh = w >> 8;
        const uint32_t b[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x64006400u,
                               (wh & 0x000F000Fu) | 0x64006400u, (wh & 0x00F000F0u) | 0x64006400u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 h = *reinterpret_cast<const __half2*>(&b[j]);
            const __half2 q = (j & 1) ? __hfma2(h, sixteenth, m72) : __hsub2(h, off);   // exact
            const __half2 v = __hmul2(q, s);
            r[4 * c + j] = *reinterpret_cast<const uint32_t*>(&v);
        }
    }
}

// Descriptor step (16-byte units) from a stage's first K step to step j:
// K block j / 4 (bsub: its size in 16-byte units), 32 (j % 4) bytes into
// its 128-byte rows.
__device__ __forceinline__ uint64_t sab_boff(int j, uint32_t bsub) {
    return uint64_t(uint32_t(j >> 2) * bsub + 2u * uint32_t(j & 3));
}

// Accumulators of a tile with npad token columns: two (one per MMA warp,
// alternate K steps) when both fit one 128-column buffer, else one.
__host__ __device__ inline int sab_accumulators(int npad) { return npad <= 64 ? 2 : 1; }

// Bounded wait that also gives up early once a timed-out wait has been
// latched (STRATA_ETIMEOUT), so one failed wait in the grid does not leave
// every later wait to run out its full limit.
__device__ __forceinline__ bool sab_wait(uint64_t* bar, uint32_t parity, const uint32_t* err) {
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *reinterpret_cast<const volatile uint32_t*>(err) == 4u)
            return false;
    }
    return false;
}

// Position of element e (within its group of 8) in the MMA order above.
__device__ __forceinline__ int mma_pos(int i) {
    const int e = i & 7;
    return (i & ~7) | ((e & 3) * 2 + (e >> 2));
}

template <int MODE>
__global__ void __launch_bounds__(kSabThreads, 1)
    k_pf_gemm_sab(const __grid_constant__ SabXMaps map_x, const __grid_constant__ SabXMaps map_x2,
                  const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_ws,
                  const __grid_constant__ CUtensorMap map_w2,
                  const __grid_constant__ CUtensorMap map_ws2, GemmLaunch a) {
    extern __shared__ uint8_t sab_dyn[];
    // full: a stage's activations landed (the producer's arrival with the
    // transaction bytes) and its A stage written (128 dequantisation
    // arrivals); empty: its MMAs done (activations and A stage both free
    // again).  Every waiter of a barrier waits for each of its phases in
    // turn: the parity waits below are only sound that way.
    __shared__ __align__(8) uint64_t full[kSabStages], empty[kSabStages];
    __shared__ __align__(8) uint64_t wfull[kSabWStages], wempty[kSabWStages];
    __shared__ __align__(8) uint64_t sc_full[2], sc_empty[2], acc_full[2], acc_empty[2];
    __shared__ __align__(8) uint64_t mma_done;
    __shared__ uint32_t tmem_base;
    __shared__ int s_ntiles;
    __shared__ uint32_t s_range;       // an fp16 output left the finite range
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sab_dyn) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t scb = sab_scale_bytes(a.K_max);
    uint8_t* w_base = base + size_t(kSabStages) * kSabStageBytes;   // weight stages
    uint8_t* sc_base = w_base + size_t(kSabWStages) * kSabWBytes;   // two scale buffers

    pdl_launch();
    if (tid == 0) {
        for (int i = 0; i < kSabStages; ++i) {
            mbar_init(&full[i], 1 + 128);
            mbar_init(&empty[i], kSabMmaWarps);
        }
        for (int i = 0; i < kSabWStages; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], 128);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sc_full[i], 1);
            mbar_init(&sc_empty[i], 128 * kSabDeqSets);
            mbar_init(&acc_full[i], kSabMmaWarps);
            mbar_init(&acc_empty[i], 128);
        }
        mbar_init(&mma_done, kSabMmaWarps);
        mbar_fence_init();
        s_range = 0u;
        for (int i = 0; i < kSabXMaps; ++i) tma_prefetch_map(&map_x.m[i]);
        tma_prefetch_map(&map_w);
    }
    if (wid == 1) {
        tmem_alloc(&tmem_base, kSabTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    if (tid == 0) s_ntiles = __ldcg(a.n_mblocks) * a.nb_max;
    __syncthreads();
    const int n_tiles = s_ntiles;
    const uint32_t tmem = tmem_base;

    // The CTAs take the tiles in rounds of gridDim.x, alternate rounds in
    // reverse CTA order: with the block list largest first, the CTAs that
    // drew the larger tiles of one round draw the smaller ones of the next.
    // A CTA's tile grows with its round, so the first past n_tiles ends it.
    auto tile_at = [&](int r) {
        const int G = int(gridDim.x), b = int(blockIdx.x);
        return r * G + ((r & 1) ? G - 1 - b : b);
    };
    // tile -> (token block, 128-row weight tile); false when the weight tile
    // does not exist for the block's group
    // Every role reads the next tile's block entry one tile ahead, so its L2
    // round trip overlaps the current tile.
    auto fetch = [&](int tile) {
        MBlock m{0, 0, 0, 0};
        if (tile < n_tiles) {
            const int4 v = __ldcg(reinterpret_cast<const int4*>(a.mblocks) + tile / a.nb_max);
            m = MBlock{v.x, v.y, v.z, v.w};
        }
        return m;
    };
    auto tile_info = [&](int tile, const MBlock& m, int& g, int& row, int& nrows, int& mt, int& W,
                         int& K) {
        mt = tile % a.nb_max;
        g = m.group;
        row = m.row;
        nrows = m.nrows;
        const bool sh = g == a.E;
        W = sh ? a.N2 : a.N;
        K = sh ? a.K2 : a.K;
        return mt * kBM < W && nrows > 0;
    };

    if (wid == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kst = 0, ti = 0;               // pipeline stages and tiles so far
            uint32_t ws = 0, wph = 0;               // weight ring slot and phase
            uint32_t wcount = 0;                     // weight stages so far
            MBlock mb_next = fetch(tile_at(0));
            for (int r = 0, tile = tile_at(0); tile < n_tiles; tile = tile_at(++r)) {
                const MBlock mb = mb_next;
                mb_next = fetch(tile_at(r + 1));
                int g, row, nrows, mt, W, K;
                if (!tile_info(tile, mb, g, row, nrows, mt, W, K)) continue;
                const bool sh = g == a.E;
                const int nbox = (nrows + kSabBoxRows - 1) / kSabBoxRows;
                const CUtensorMap* mx = &((sh && MODE == kGemmDown) ? map_x2 : map_x).m[nbox - 1];
                const CUtensorMap* mw = sh ? &map_w2 : &map_w;
                const CUtensorMap* mws = sh ? &map_ws2 : &map_ws;
                const int xrow = (sh && MODE == kGemmGateUp) ? a.a_shared_row0 + row : row;
                const int wrow = (sh ? 0 : g * W) + mt * kBM;
                const uint32_t buf = ti & 1u, sround = ti >> 1;
                if (sround > 0 && !sab_wait(&sc_empty[buf], (sround - 1) & 1, a.err))
                    latch_timeout(a.err, 31, buf, sround, tile);
                mbar_expect_tx(&sc_full[buf], uint32_t(kBM) * uint32_t(K / 32) * 2u);
                tma_load_3d(sc_base + buf * scb, mws, 0, wrow, 0, &sc_full[buf]);
                const uint32_t xbytes = uint32_t(nbox) * (kSabBoxRows * 128u) * uint32_t(kSabKS / 64);
                const int nks = K / kSabKS;
                for (int ks = 0; ks < nks; ++ks, ++kst) {
                    {
                        // one weight stage: this pipeline stage
                        if (kst >= uint32_t(kSabWStages) && !sab_wait(&wempty[ws], wph ^ 1u, a.err))
                            latch_timeout(a.err, 30, ws, kst, tile);
                        mbar_expect_tx(&wfull[ws], kSabWBytes);
                        tma_load_2d(w_base + ws * kSabWBytes, mw, ks * (kSabKS / 2), wrow,
                                    &wfull[ws]);
                        ++wcount;
                        if (++ws == uint32_t(kSabWStages)) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    }
                    const uint32_t s = kst & (kSabStages - 1), round = kst / kSabStages;
                    if (round > 0 && !sab_wait(&empty[s], (round - 1) & 1, a.err))
                        latch_timeout(a.err, 32, s, round, tile);
                    uint8_t* st = base + s * kSabStageBytes;
                    mbar_expect_tx(&full[s], xbytes);
                    tma_load_3d(st, mx, 0, xrow, (kSabKS / 64) * ks, &full[s]);
                }
                ++ti;
            }
            // Every copy has landed before the CTA exits, also when a wait
            // gave up: the last round of each slot (completed long ago when
            // nothing failed).
            for (uint32_t i = 0; i < uint32_t(kSabStages) && i < kst; ++i) {
                const uint32_t k = kst - 1 - i;
                mbar_wait(&full[k % kSabStages], (k / kSabStages) & 1);
            }
            for (uint32_t i = 0; i < uint32_t(kSabWStages) && i < wcount; ++i) {
                const uint32_t k = wcount - 1 - i;
                mbar_wait(&wfull[k % kSabWStages], (k / kSabWStages) & 1);
            }
            for (uint32_t i = 0; i < 2u && i < ti; ++i) {
                const uint32_t t = ti - 1 - i;
                mbar_wait(&sc_full[t & 1u], (t >> 1) & 1);
            }
        }
    } else if (wid <= kSabMmaWarps) {
        // ----------------------------------------------------------- MMA
        if (lane == 0) {
            const int mw = wid - 1;          // with two accumulators: K steps j % 2 == mw
            uint32_t kst = 0, ti = 0;
            MBlock mb_next = fetch(tile_at(0));
            for (int r = 0, tile = tile_at(0); tile < n_tiles; tile = tile_at(++r)) {
                const MBlock mb = mb_next;
                mb_next = fetch(tile_at(r + 1));
                int g, row, nrows, mt, W, K;
                if (!tile_info(tile, mb, g, row, nrows, mt, W, K)) continue;
                const uint32_t dbuf = ti & 1u, dround = ti >> 1;
                if (dround > 0 && !sab_wait(&acc_empty[dbuf], (dround - 1) & 1, a.err))
                    latch_timeout(a.err, 33, dbuf, dround, tile);
                tc_fence_after();
                const int npad = (nrows + 15) & ~15;
                const int nacc = sab_accumulators(npad);
                const uint32_t idesc = idesc_f16(kBM, npad, 0);
                // the stage's second K block follows the first's box rows
                const uint32_t bsub = uint32_t((nrows + kSabBoxRows - 1) / kSabBoxRows) *
                                      (kSabBoxRows * 128u / 16u);
                const uint32_t d_tmem = tmem + dbuf * kSabDCols + uint32_t(mw * (kSabDCols / 2));
                const int nks = K / kSabKS;
                for (int ks = 0; ks < nks; ++ks, ++kst) {
                    const uint32_t s = kst & (kSabStages - 1), round = kst / kSabStages;
                    if (!sab_wait(&full[s], round & 1, a.err))
                        latch_timeout(a.err, 34, s, round, tile);
                    tc_fence_after();
                    // the stage's first K step; step j is sub-block j / 4 of B,
                    // 32 (j % 4) bytes into its rows, and A columns 8 j on
                    const uint64_t b0 = sdesc_k_sw128(smem_u32(base + s * kSabStageBytes));
                    const uint32_t a0 = tmem + uint32_t(kSabACol0) + s * kSabACols;
                    if (nacc == 1) {
                        if (mw == 0) {
#pragma unroll
                            for (int j = 0; j < kSabKS / 16; ++j)
                                umma_f16_tmem_a(d_tmem, a0 + uint32_t(8 * j), b0 + sab_boff(j, bsub),
                                                idesc, (ks | j) != 0 ? 1u : 0u);
                        }
                    } else {
                        const uint64_t bm = b0 + uint64_t(2 * mw);     // + 32 bytes on odd steps
                        const uint32_t am = a0 + uint32_t(8 * mw);
#pragma unroll
                        for (int jj = 0; jj < kSabKS / 32; ++jj)
                            umma_f16_tmem_a(d_tmem, am + uint32_t(16 * jj), bm + sab_boff(2 * jj, bsub),
                                            idesc, (ks | jj) != 0 ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);
                }
                umma_commit(&acc_full[dbuf]);
                ++ti;
            }
            // no product may still be writing the TMEM when it is freed
            umma_commit(&mma_done);
            mbar_wait(&mma_done, 0);
        }
    } else if (wid < kSabDeq0 + 4 * kSabDeqSets) {
        // ------------------------------------------------ dequantisation
        const int q = wid & 3;                 // TMEM lane quarter
        const int m = q * 32 + lane;           // weight row of the tile
        const uint32_t set = uint32_t(wid - kSabDeq0) >> 2;   // this set's stages: kst % 2 == set
        uint32_t kst = 0, ti = 0;
        uint32_t ws = 0, wph = 0;
        MBlock mb_next = fetch(tile_at(0));
        for (int r = 0, tile = tile_at(0); tile < n_tiles; tile = tile_at(++r)) {
            const MBlock mb = mb_next;
            mb_next = fetch(tile_at(r + 1));
            int g, row, nrows, mt, W, K;
            if (!tile_info(tile, mb, g, row, nrows, mt, W, K)) continue;
            const uint32_t buf = ti & 1u, sround = ti >> 1;
            if (!sab_wait(&sc_full[buf], sround & 1, a.err))
                latch_timeout(a.err, 36, buf, sround, tile);
            const uint32_t scrow = smem_u32(sc_base + buf * scb) + uint32_t(m * 16);
            const int nks = K / kSabKS;
            for (int ks = 0; ks < nks; ++ks, ++kst) {
                const uint32_t cws = ws, cwph = wph;
                if (++ws == uint32_t(kSabWStages)) {
                    ws = 0;
                    wph ^= 1u;
                }
                if ((kst & 1u) != set) continue;
                const uint32_t s = kst & (kSabStages - 1), round = kst / kSabStages;
                if (!sab_wait(&wfull[cws], cwph, a.err)) latch_timeout(a.err, 37, cws, kst, tile);
                const uint32_t wrow_s = smem_u32(w_base + cws * kSabWBytes) + uint32_t(m * 128);
                // the stage's 8 scales (two a 64-wide sub-block)
                const uint4 sc8 = lds128(scrow + uint32_t(ks) * (kBM * 16u));
                const uint32_t scw[4] = {sc8.x, sc8.y, sc8.z, sc8.w};
                if (round > 0 && !sab_wait(&empty[s], (round - 1) & 1, a.err))
                    latch_timeout(a.err, 38, s, round, tile);
                tc_fence_after();
#pragma unroll
                for (int sb = 0; sb < kSabKS / 64; ++sb) {
                    // 32 bytes of row m: 16-byte chunks c, c + 1 of the swizzled row
                    const int c = sb * 2;
                    const uint4 w0 = lds128(wrow_s + uint32_t(((c ^ (m & 7)) & 7) * 16));
                    const uint4 w1 = lds128(wrow_s + uint32_t((((c + 1) ^ (m & 7)) & 7) * 16));
                    uint32_t r[32];
                    dequant_row_regs(w0, w1, scw[sb], r);
                    tmem_st32(tmem + (uint32_t(q * 32) << 16) + uint32_t(kSabACol0) +
                                  s * kSabACols + uint32_t(32 * sb),
                              r);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&full[s]);
                mbar_arrive(&wempty[cws]);
            }
            mbar_arrive(&sc_empty[buf]);
            ++ti;
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int q = wid & 3;
        const int m = q * 32 + lane;           // weight row of the tile
        uint32_t ti = 0;
        MBlock mb_next = fetch(tile_at(0));
        for (int r = 0, tile = tile_at(0); tile < n_tiles; tile = tile_at(++r)) {
            const MBlock mb = mb_next;
            mb_next = fetch(tile_at(r + 1));
            int g, row, nrows, mt, W, K;
            if (!tile_info(tile, mb, g, row, nrows, mt, W, K)) continue;
            const bool sh = g == a.E;
            const uint32_t dbuf = ti & 1u, dround = ti >> 1;
            if (!sab_wait(&acc_full[dbuf], dround & 1, a.err))
                latch_timeout(a.err, 39, dbuf, dround, tile);
            tc_fence_after();
            const uint32_t tl = tmem + (uint32_t(q * 32) << 16) + dbuf * kSabDCols;
            const bool two = sab_accumulators((nrows + 15) & ~15) == 2;
            for (int c0 = 0; c0 < nrows; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tl + uint32_t(c0), v);
                if (two) {
                    // the odd K steps' accumulator, 64 columns on
                    uint32_t v1[32];
                    tmem_ld32(tl + uint32_t(kSabDCols / 2 + c0), v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                } else {
                    tmem_ld_wait();
                }
                const int nv = min(32, nrows - c0);
                uint32_t inf_nan = 0u;    // an fp16 operand left the finite range
                if (MODE == kGemmGateUp) {
                    // rows 2i (gate) and 2i + 1 (up) are lanes l and l + 1, each
                    // with every token.  One exchange per token pair gives the
                    // even lane token j's (gate, up) and the odd lane token
                    // j + 1's, so every lane computes a SwiGLU.  h is rounded to
                    // fp16 for the down product, so the fast exp and divide
                    // (relative error ~1e-6) cost nothing in accuracy.
                    const int odd = lane & 1;
                    const int i = (mt * kBM + m) >> 1;       // SwiGLU index of the pair
                    const int ld = sh ? a.ld2 : a.ldo;
                    const size_t r0 = size_t(row + c0 + odd) * ld;
                    __half* hb = (sh ? a.out2_f16 : a.out_f16) + r0 + mma_pos(i);
                    float* hf = (!sh && a.out_f32 != nullptr) ? a.out_f32 + r0 + i : nullptr;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float keep = __uint_as_float(odd ? v[j + 1] : v[j]);
                        const float send = __uint_as_float(odd ? v[j] : v[j + 1]);
                        const float other = __shfl_xor_sync(0xffffffffu, send, 1);
                        const float gt = odd ? other : keep, up = odd ? keep : other;
                        if (j + odd < nv) {
                            const float h = __fdividef(gt, 1.0f + __expf(-gt)) * up;
                            const __half hh = __float2half_rn(h);
                            inf_nan |= f16x2_not_finite(__half_as_ushort(hh));
                            hb[size_t(j) * ld] = hh;
                            if (hf != nullptr) hf[size_t(j) * ld] = h;
                        }
                    }
                    // rare: an element overflowed; the thread rewrites its own
                    // stores saturated (kept out of the loop above, which a
                    // branch per element slowed by a third)
                    if (inf_nan != 0u)
                        for (int j = odd; j < nv; j += 2) {
                            const uint32_t hu = __half_as_ushort(hb[size_t(j) * ld]);
                            hb[size_t(j) * ld] = __ushort_as_half(uint16_t(f16x2_saturate(hu)));
                        }
                } else {
                    const int o = mt * kBM + m;              // output feature
                    const size_t ld = size_t(a.ldo);
                    const size_t r0 = size_t(row + c0) * ld + o;
                    if (!sh && a.out_bf16 != nullptr) {
                        uint16_t* yb = a.out_bf16 + r0;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nv) yb[j * ld] = f32_to_bf16(__uint_as_float(v[j]));
                    } else {
                        __half* yh = (sh ? a.out2_f16 : a.out_f16) + r0;
#pragma unroll
                        // no range check here: this epilogue paces the down
                        // products (a check per element cost a quarter of the
                        // kernel); y is no tensor-core operand, and the
                        // combine checks the outputs it makes of it
                        for (int j = 0; j < 32; ++j)
                            if (j < nv) yh[j * ld] = __float2half_rn(__uint_as_float(v[j]));
                    }
                }
                if (inf_nan != 0u) s_range = 1u;       // latched once, at the end
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[dbuf]);
            ++ti;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (wid == 1) tmem_dealloc(tmem, kSabTmemCols);
    if (tid == 0 && s_range != 0u) latch(a.err, STRATA_ERANGE);
}

// ------------------------------------------------------------------ host
bool prefill_gemm_fits(int K_max) { return sab_smem_bytes(K_max) <= kPfSmemBudget; }

namespace {

PFN_cuTensorMapEncodeTiled_v12000 sab_encode_fn() {
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
bool sab_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
             uint64_t rows, uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
    auto fn = sab_encode_fn();
    if (fn == nullptr || base == nullptr) return false;
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

// Scale map of a row-major [rows][K / 32] fp16 array viewed as (8 scales,
// rows, K / 256 groups); the box (8, 128, K / 256) is one tile's scales.
bool sab_scale_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows) {
    auto fn = sab_encode_fn();
    if (fn == nullptr || base == nullptr) return false;
    const cuuint64_t gdim[3] = {8, rows, K / 256};
    const cuuint64_t gstride[2] = {K / 16, 16};
    const cuuint32_t box[3] = {8, cuuint32_t(kBM), cuuint32_t(K / 256)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), gdim, gstride, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activation maps of a row-major [rows][K] fp16 array viewed as (64
// elements, rows, K / 64 blocks): the box (64, 32 (i + 1), 2) lands as two
// 64-wide K blocks one after the other, each with the 128-byte swizzle.
bool sab_xmaps(SabXMaps* m, const void* base, uint64_t K, uint64_t rows) {
    auto fn = sab_encode_fn();
    if (fn == nullptr || base == nullptr) return false;
    const cuuint64_t gdim[3] = {uint64_t(kBK), rows, K / kBK};
    const cuuint64_t gstride[2] = {K * 2, uint64_t(kBK) * 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    for (int i = 0; i < kSabXMaps; ++i) {
        const cuuint32_t box[3] = {cuuint32_t(kBK), cuuint32_t(kSabBoxRows * (i + 1)),
                                   cuuint32_t(kSabKS / kBK)};
        if (fn(&m->m[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), gdim,
               gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

template <int MODE>
cudaError_t run_sab(GemmLaunch g, const SabXMaps& mx, const SabXMaps& mx2,
                    const CUtensorMap& mw, const CUtensorMap& mws, const CUtensorMap& mw2,
                    const CUtensorMap& mws2, cudaStream_t s) {
    const Dev d = device_info();
    const size_t dyn = sab_smem_bytes(g.K_max);
    if (dyn > kPfSmemBudget || g.K % 256 != 0 || g.K2 % 256 != 0) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_pf_gemm_sab<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.sms);
    cfg.blockDim = dim3(kSabThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_pf_gemm_sab<MODE>, mx, mx2, mw, mws, mw2, mws2, g);
    if (e == cudaSuccess) prof_after_launch(s);
    return e;
}

}  // namespace

cudaError_t launch_prefill_gate_up(const PfExperts& p, cudaStream_t s) {
    const int H = p.H, I = p.I, Is = p.Is, E = p.E;
    // activations xg [xg_rows][H]; weights: packed rows and their scales in
    // 128-row boxes.  A weight set the block list cannot name gets the other
    // set's maps.
    SabXMaps mx;
    CUtensorMap mq, ms, mq2, ms2;
    if (!sab_xmaps(&mx, p.xg, H, p.xg_rows)) return cudaErrorInvalidValue;
    if (p.routed &&
        (!sab_map(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.gu_q, H / 2, uint64_t(E) * 2 * I,
                  kSabWRowBytes, kBM, true) ||
         !sab_scale_map(&ms, p.gu_s, H, uint64_t(E) * 2 * I)))
        return cudaErrorInvalidValue;
    if (p.shared &&
        (!sab_map(&mq2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.sh_gu_q, H / 2, 2 * Is,
                  kSabWRowBytes, kBM, true) ||
         !sab_scale_map(&ms2, p.sh_gu_s, H, 2 * Is)))
        return cudaErrorInvalidValue;
    if (!p.routed) {
        mq = mq2;
        ms = ms2;
    }
    if (!p.shared) {
        mq2 = mq;
        ms2 = ms;
    }
    GemmLaunch g{};
    g.N = 2 * I;
    g.N2 = 2 * Is;
    g.K = H;
    g.K2 = H;
    g.K_max = H;
    g.E = E;
    g.mblocks = p.mblocks;
    g.n_mblocks = p.n_mblocks;
    g.nb_max = (2 * (I > Is ? I : Is)) / kBM;
    g.a_shared_row0 = p.xg_shared_row0;
    g.out_f16 = p.h;
    g.out_f32 = p.h_f32;
    g.ldo = I;
    g.out2_f16 = p.hs;
    g.ld2 = Is;
    g.err = p.err;
    return run_sab<kGemmGateUp>(g, mx, mx, mq, ms, mq2, ms2, s);
}

cudaError_t launch_prefill_down(const PfExperts& p, cudaStream_t s) {
    const int T = p.T, K = p.K, H = p.H, I = p.I, Is = p.Is, E = p.E;
    // activations h [T*K][I] (routed) or hs [T][Is] (shared)
    SabXMaps mx, mx2;
    CUtensorMap mq, ms, mq2, ms2;
    if (p.routed &&
        (!sab_xmaps(&mx, p.h, I, uint64_t(T) * K) ||
         !sab_map(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.dn_q, I / 2, uint64_t(E) * H,
                  kSabWRowBytes, kBM, true) ||
         !sab_scale_map(&ms, p.dn_s, I, uint64_t(E) * H)))
        return cudaErrorInvalidValue;
    if (p.shared &&
        (!sab_xmaps(&mx2, p.hs, Is, T) ||
         !sab_map(&mq2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.sh_dn_q, Is / 2, H,
                  kSabWRowBytes, kBM, true) ||
         !sab_scale_map(&ms2, p.sh_dn_s, Is, H)))
        return cudaErrorInvalidValue;
    if (!p.routed) {
        mx = mx2;
        mq = mq2;
        ms = ms2;
    }
    if (!p.shared) {
        mx2 = mx;
        mq2 = mq;
        ms2 = ms;
    }
    GemmLaunch d{};
    d.N = H;
    d.N2 = H;
    d.K = I;
    d.K2 = Is;
    d.K_max = I > Is ? I : Is;
    d.E = E;
    d.mblocks = p.mblocks;
    d.n_mblocks = p.n_mblocks;
    d.nb_max = H / kBM;
    d.a_shared_row0 = 0;
    d.out_f16 = p.y;
    d.out_bf16 = p.y_bf16;
    d.out2_f16 = p.ysh;
    d.ldo = H;
    d.err = p.err;
    return run_sab<kGemmDown>(d, mx, mx2, mq, ms, mq2, ms2, s);
}

}  // namespace strata
