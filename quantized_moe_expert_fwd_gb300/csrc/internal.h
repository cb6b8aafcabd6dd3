// internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/strata_moe.h"

namespace strata {

constexpr int kDecodeMaxTokens = 32;
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kDownRowsPerCta = 14;

// Byte offsets of the workspace regions for a call with T tokens.  Every
// region starts on a 256-byte boundary; the control block is at 0.
struct WsLayout {
    size_t ctl, logits, ids, w, sig, counts, offsets, perm, inv, h, hs, x, out, total;
    // prefill (T > kDecodeMaxTokens)
    size_t tiles, xf16, hf16, y, shy;
};

WsLayout ws_layout(const strata_moe_dims& d, int T);

struct Dev {
    int sms;
};
Dev device_info();

// -------------------------------------------------------------- launchers
struct RouteLaunch {
    const uint16_t* router; const float* bias;
    const uint16_t* x;
    float* logits;                    // ws [T][E+1]
    const uint8_t* shq; const uint16_t* shs; float* hs; int Is; int do_shared;
    int do_select;
    int32_t* ids; float* w; float* sig;                 // ws copies
    int32_t* ids_user; float* w_user; float* sig_user; float* logits_user;
    const int32_t* ids_in; const float* w_in;           // forced routing
    int do_permute;
    int32_t* counts; int32_t* offsets; int32_t* perm; int32_t* inv;
    void* ctl;
    int T, H, E, K;
};
cudaError_t launch_route_decode(const RouteLaunch& a, cudaStream_t s);

struct GuLaunch {
    const uint8_t* q; const uint16_t* sc;
    const uint16_t* x;
    const int32_t* offsets; const int32_t* perm;
    float* h;
    uint32_t* err;
    int T, H, I, E, K;
    int shared;
};
cudaError_t launch_gate_up_decode(const GuLaunch& a, cudaStream_t s);

enum DownMode { kDownFused = 0, kDownSlots = 1, kDownCombine = 2 };
struct DownLaunch {
    const uint8_t* q; const uint16_t* sc;
    const uint8_t* shq; const uint16_t* shs;
    const float* h; const float* hs;
    const int32_t* offsets; const int32_t* inv;
    const float* w; const float* sig;
    const uint16_t* y_in; uint16_t* y_out;
    uint16_t* out; float* resid;
    uint32_t* err;
    int T, H, I, Is, E, K;
    int mode;
};
cudaError_t launch_down_decode(const DownLaunch& a, cudaStream_t s);

cudaError_t launch_rmsnorm(const float* r, int T, int H, float eps, uint16_t* x, cudaStream_t s);

}  // namespace strata

namespace strata {
cudaError_t launch_permute_small(const int32_t* ids, int T, int K, int E, int32_t* counts,
                                 int32_t* offsets, int32_t* perm, int32_t* inv, uint32_t* err,
                                 cudaStream_t s);
}  // namespace strata
