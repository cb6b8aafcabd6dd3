// internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda_fp16.h>

#include "../../include/strata_moe.h"

namespace strata {

constexpr int kDecodeMaxTokens = 32;       // the decode kernels take up to this many tokens
// A whole layer (layer, block and stack calls) runs on the decode kernels up
// to this many tokens and on the tensor-core kernels above, when the layer's
// shape allows them: measured on GB300, the decode kernels' cost grows by
// ~16 us a token, the tensor-core path's by ~2 us on a ~45 us base, equal at 2.
constexpr int kLayerDecodeMaxTokens = 2;
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kDownRowsPerCta = 16;
// shared-memory rings of the decode expert kernels
constexpr int kGuMaxStages = 8;
constexpr size_t kGuRingBytes = 147456;   // 4 stages of 16 gate/up row pairs at H = 2048
constexpr size_t kGuSmemBytes = 196608;   // ring + the tokens' activations (dynamic part)
constexpr int kDnMaxStages = 24;
constexpr size_t kDnRingBytes = 114688;
// plan: [0] touched experts, header pad, then e[E], off[E], cnt[E], tok[T*K]
constexpr int kPlanHeader = 4;

// prefill (T > kDecodeMaxTokens) tiles: 128 rows x 64 K per stage
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr size_t kPfSmemBudget = 225280;
constexpr int kRouterSplitMax = 8;       // K slices of the prefill router GEMM
enum GemmMode { kGemmGateUp = 1, kGemmDown = 2 };

// One block of up to 128 rows of one group (a routed expert, or the shared
// expert as group E) for the prefill GEMMs.  row: first row of the group's
// A operand space (a slot for routed experts, a token for the shared one).
struct MBlock {
    int group, row, nrows, pad;
};

// Byte offsets of the workspace regions for a call with T tokens.  Every
// region starts on a 256-byte boundary; the control block is at 0.  The
// decode regions (plan, h, hs as fp32) exist for T <= kDecodeMaxTokens and
// end at decode_end; the persistent kernel's tagged exchanges follow for
// T <= kPersistMaxTokens, the prefill ones (per-block counts, row blocks,
// fp16 operands, bf16 outputs) for T > kLayerDecodeMaxTokens.
struct WsLayout {
    size_t ctl, flags, logits, ids, w, sig, counts, offsets, perm, inv, plan, h, hs, x, out;
    size_t cnt_blk, base_blk, mblocks, n_mblocks, lgp, xg, h16, hs16, y, ysh;
    size_t ll_logits, ll_hs, ll_h, ll_resid;   // persistent kernel (T <= kPersistMaxTokens)
    size_t decode_end, total;
};

WsLayout ws_layout(const strata_moe_dims& d, int T);

struct Dev {
    int sms;
};
Dev device_info();

// Called after every kernel launch: when moe_layer_profile is running on
// this host thread, records a CUDA event on the launch's stream.
void prof_after_launch(cudaStream_t s);

// -------------------------------------------------------------- launchers
struct RouteLaunch {
    const uint16_t* router; const float* bias;
    const uint16_t* x;
    float* logits;                    // ws [T][E+1]
    const uint8_t* shq; const uint16_t* shs; float* hs; int Is; int do_shared;
    int do_select;                    // 0: only the shared-gate row (forced routing)
    int T, H, E, K;
};
cudaError_t launch_route_decode(const RouteLaunch& a, cudaStream_t s);

struct SelectLaunch {
    const float* logits;
    int32_t* ids; float* w; float* sig; float* logits_out;
    uint32_t* err;
    int T, E, K;
};
cudaError_t launch_select(const SelectLaunch& a, cudaStream_t s);

enum GuMode { kGuRoute = 0, kGuPlan = 1, kGuShared = 2 };
struct GuLaunch {
    const uint8_t* q; const uint16_t* sc;
    const uint16_t* x;
    // kGuRoute: routing from logits (or forced ids/w), published by CTA 0
    const float* logits;
    const int32_t* forced_ids; const float* forced_w;
    int32_t* ids; float* w; float* sig;
    int32_t* ids_user; float* w_user; float* sig_user;
    int32_t* counts; int32_t* offsets; int32_t* perm; int32_t* inv; int32_t* plan_out;
    // kGuPlan: plan built by k_plan
    const int32_t* plan;
    float* h;
    uint32_t* err;
    int T, H, I, E, K;
    int mode;
    int tail_skip;                    // kGuRoute: 0 off, else leave out experts every token
                                      // ranks past this place (1 <= tail_skip < K)
    int stages, x_smem;               // set by the launcher
};
cudaError_t launch_gate_up_decode(GuLaunch a, cudaStream_t s);

enum DownMode { kDownFused = 0, kDownSlots = 1, kDownCombine = 2 };
struct DownLaunch {
    const uint8_t* q; const uint16_t* sc;
    const uint8_t* shq; const uint16_t* shs;
    const float* h; const float* hs;
    const int32_t* plan; const int32_t* inv;
    const float* w; const float* sig;
    const uint16_t* y_in; uint16_t* y_out;
    uint16_t* out; float* resid;
    uint32_t* err;
    int T, H, I, Is, E, K;
    int mode;
    int stages;                       // set by the launcher
};
cudaError_t launch_down_decode(DownLaunch a, cudaStream_t s);

cudaError_t launch_plan(const int32_t* offsets, const int32_t* perm, int T, int K, int E,
                        int32_t* plan, uint32_t* err, cudaStream_t s);
cudaError_t launch_permute_small(const int32_t* ids, int T, int K, int E, int32_t* counts,
                                 int32_t* offsets, int32_t* perm, int32_t* inv, uint32_t* err,
                                 cudaStream_t s);
cudaError_t launch_rmsnorm(const float* r, int T, int H, float eps, uint16_t* x, cudaStream_t s);

// ------------------------------------------------ persistent decode layers
// A whole decode-size layer (or a stack of residual layers) as one launch of
// one CTA per SM (persist.cu).
// Tokens a whole-layer call it takes: one.  At T = 1 (2048-hidden,
// 256-expert, top-8 layers rotating in a CUDA graph) it takes 19.4 us against
// 32.2 for the three decode kernels.  Calls of 2 and 3 tokens ended in a
// launch failure in a crossover measurement after the kernel was tuned for
// one token (its 15-stage gate/up ring then wraps within a layer); the cause
// was not found by reading the code, so the kernel takes no more than one.
constexpr int kPersistMaxTokens = 1;
constexpr int kPersistTokensCap = 1;
constexpr int kMaxGrid = 1024;            // grid barrier flags in the workspace
constexpr int kPxMaxLayers = 40;          // layers one launch carries
// 1 producer + 15 consumer warps (128 registers a thread): the int4 dot
// products keep the ALU pipes busy only with several warps on each of the
// SM's four sub-partitions
constexpr int kPxConsumers = 15;
constexpr int kPxRowPairs = 2;            // gate/up row pairs per ring stage (one warp's)
constexpr int kPxGuMaxStages = 15;
constexpr int kPxDnMaxStages = 32;
constexpr size_t kPxSmemBudget = 200 * 1024;   // dynamic shared memory at most
constexpr size_t kPxSmemMin = 120 * 1024;      // at least: one CTA per SM

struct PxLayer {
    const uint16_t* router; const float* bias;
    const uint8_t* gu_q; const uint16_t* gu_s;
    const uint8_t* dn_q; const uint16_t* dn_s;
    const uint8_t* sh_gu_q; const uint16_t* sh_gu_s;
    const uint8_t* sh_dn_q; const uint16_t* sh_dn_s;
};

// Launch geometry: down rows a CTA owns, ring depths, dynamic shared memory
// offsets (bytes, 128-aligned) and stage sizes.
struct PxGeo {
    int MC, R, gu_stages, dn_stages;
    uint32_t off_x, off_r, off_sd, off_d, off_y, off_g;
    uint32_t sd_q, sd_bytes, d_q, d_stage, g_q, g_stage, dyn;
};

struct PxArgs {
    int T, H, E, K, I, Is, n_layers;
    float eps;
    const uint16_t* x_in;            // resid == NULL (one layer): bf16 [T][H]
    float* resid;                    // fp32 [T][H]: each layer normalises it, adds its output
    uint16_t* out;                   // the last layer's bf16 output [T][H], or NULL
    uint16_t* x_out;                 // the last layer's normalised input [T][H], or NULL
    const int32_t* forced_ids;       // [n_layers][T][K] or NULL
    const float* forced_w;
    int32_t* ids_user; float* w_user; float* sig_user;   // the last layer's routing, or NULL
    // workspace: the cross-CTA exchanges as tagged 64-bit words (value low,
    // tag high): logits [T][E+1], shared SwiGLU [T][Is], routed SwiGLU
    // [T*K][I] in slot order, the stack's residual [T][H]
    uint64_t* ll_logits; uint64_t* ll_hs; uint64_t* ll_h; uint64_t* ll_resid;
    int32_t* ids; float* w; float* sig;
    int32_t* counts; int32_t* offsets; int32_t* perm; int32_t* inv;
    uint32_t* flags; uint32_t* err;
    uint32_t grid_wait_limit;        // polls before a grid barrier gives up
    int R, gu_stages, dn_stages;
    uint32_t off_x, off_r, off_sd, off_d, off_y, off_g;
    uint32_t sd_q, sd_bytes, d_q, d_stage, g_q, g_stage;
    PxLayer L[kPxMaxLayers];
};

// Whether the persistent kernel takes this shape at T tokens on a grid of G
// CTAs (resid: the calls that normalise a residual in the kernel), and its
// geometry.
bool px_geometry(const strata_moe_dims& d, int T, bool forced, bool resid, int G, PxGeo* g);
cudaError_t launch_persistent(const PxArgs& a, const PxGeo& g, cudaStream_t s);

// Phase timestamps of the persistent kernel, recorded only by a library
// built with STRATA_PX_TRACE (the default build has none): per CTA, for the
// last launch's layers 0, 1, n/2 and n-1 (slots 0..3), kPxTracePoints
// global-timer readings (ns), the points of strata_px_trace_read.
constexpr int kPxTraceSlots = 4;
constexpr int kPxTracePoints = 16;
constexpr size_t kPxTraceBytes = size_t(kMaxGrid) * kPxTraceSlots * kPxTracePoints * 8;
// Copies the timestamps to host memory; cudaErrorNotSupported without tracing.
cudaError_t px_trace_copy(void* host, size_t bytes);
// polls before a grid barrier of the persistent kernel gives up (testing
// hook, strata_set_grid_wait_limit; 0: the default)
uint32_t grid_wait_limit();
void set_grid_wait_limit(uint32_t polls);

// ---------------------------------------------------------------- prefill
struct PfSelectLaunch {
    const float* part; int nsplit;    // router GEMM K slices [nsplit][T][E + 1], bias in slice 0
    float* logits_user;
    const int32_t* forced_ids; const float* forced_w;
    int32_t* ids; float* w; float* sig;
    int32_t* ids_user; float* w_user; float* sig_user;
    uint32_t* err;
    int T, E, K;
};
struct PfScanLaunch {
    const int32_t* cnt_blk; int32_t* base_blk;
    int32_t* counts; int32_t* offsets;
    MBlock* mblocks; int32_t* n_mblocks;
    int nblk, E, T, with_shared;
};
struct GemmLaunch {
    const MBlock* mblocks; const int32_t* n_mblocks;
    int N, N2, K, K2, K_max;      // N, K of routed groups; N2, K2 of the shared group
    int nb_max, E, a_shared_row0;
    float* out_f32;               // gate/up: routed h also in fp32 (or NULL)
    __half* out_f16; __half* out2_f16;
    uint16_t* out_bf16; uint16_t* out2_bf16;
    int ldo, ld2;
    uint32_t* err;
};
struct PfRoute {
    const uint16_t* x; const uint16_t* router; const float* bias;
    float* part; float* logits_user;    // part: kRouterSplitMax * T * (E + 1) floats
    const int32_t* forced_ids; const float* forced_w;
    int32_t* ids; float* w; float* sig;
    int32_t* ids_user; float* w_user; float* sig_user;
    uint32_t* err;
    int T, H, E, K;
};
struct PfBucket {
    const int32_t* ids;
    int32_t* cnt_blk; int32_t* base_blk;
    int32_t* counts; int32_t* offsets; int32_t* perm; int32_t* inv;
    MBlock* mblocks; int32_t* n_mblocks;
    uint32_t* err;
    int T, K, E, with_shared;
};
struct PfExperts {
    const uint16_t* x; const int32_t* perm;
    __half* xg;
    const uint8_t* gu_q; const uint16_t* gu_s; const uint8_t* dn_q; const uint16_t* dn_s;
    const uint8_t* sh_gu_q; const uint16_t* sh_gu_s;
    const uint8_t* sh_dn_q; const uint16_t* sh_dn_s;
    const MBlock* mblocks; const int32_t* n_mblocks;
    __half* h; __half* hs;
    __half* y; __half* ysh;
    float* h_f32;          // non-NULL: routed h also in fp32, natural order, [T*K][I]
    uint16_t* y_bf16;      // non-NULL: routed y in bf16 [T*K][H] instead of fp16 y
    int routed, shared;    // weight sets the block list may name (the other's maps alias)
    int xg_rows, xg_shared_row0;   // rows of xg; first row of the shared expert's tokens
    uint32_t* err;
    int T, K, H, I, Is, E;
};
bool prefill_supported(const strata_moe_dims& d);
// the expert GEMMs' shared memory (stages and a tile's scales) fits at this K
bool prefill_gemm_fits(int K_max);
cudaError_t launch_prefill_route(const PfRoute& r, cudaStream_t s);
cudaError_t launch_prefill_bucket(const PfBucket& b, cudaStream_t s);
// block list of the routed slots from caller offsets (offsets NULL: none)
// and/or of the shared expert over the T tokens
cudaError_t launch_prefill_blocks(const int32_t* offsets, int T, int K, int E, int with_shared,
                                  MBlock* mblocks, int32_t* n_mblocks, uint32_t* err,
                                  cudaStream_t s);
// xg rows: the T*K routed slots (token perm[row] / K), then the T tokens
cudaError_t launch_prefill_gather(const uint16_t* x, const int32_t* perm, int T, int K, int H,
                                  __half* xg, int rows, uint32_t* err, cudaStream_t s);
// fp32 [n] -> fp16 in the operand order (n a multiple of 8)
cudaError_t launch_prefill_pack(const float* src, long long n, __half* dst, uint32_t* err,
                                cudaStream_t s);
cudaError_t launch_prefill_gate_up(const PfExperts& p, cudaStream_t s);
cudaError_t launch_prefill_down(const PfExperts& p, cudaStream_t s);
// gather + gate/up + down of the routed experts and the shared one
cudaError_t launch_prefill_experts(const PfExperts& p, cudaStream_t s);
// y: fp16 (y_f16) or bf16 (y_bf16), slot order; ysh fp16
cudaError_t launch_prefill_combine(const __half* y_f16, const uint16_t* y_bf16, const __half* ysh,
                                   const int32_t* inv, const float* w, const float* sig, int T,
                                   int K, int H, uint16_t* out, float* resid, uint32_t* err,
                                   cudaStream_t s);

}  // namespace strata
