// api.cu -- the C ABI of strata_moe.h: argument checks, workspace layout and
// dispatch to the decode (GEMV) or prefill (tcgen05 GEMM) kernels.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace strata {

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(const strata_moe_dims& d, int T) {
    const size_t H = d.hidden, E = d.n_experts, K = d.top_k, I = d.inter, Is = d.shared_inter;
    const size_t t = size_t(T > 0 ? T : 1);
    WsLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    L.ctl = take(sizeof(Ctl));
    L.flags = take(size_t(kMaxGrid) * 4);     // at a fixed offset: every T shares it
    L.logits = take(t * (E + 1) * 4);
    L.ids = take(t * K * 4);
    L.w = take(t * K * 4);
    L.sig = take(t * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take(t * K * 4);
    L.inv = take(t * K * 4);
    L.x = take(t * H * 2);
    L.out = take(t * H * 2);
    if (T <= kDecodeMaxTokens) {
        L.plan = take((kPlanHeader + 3 * E + t * K) * 4);
        L.h = take(t * K * I * 4);
        L.hs = take(t * Is * 4);
    }
    L.decode_end = o;
    if (T <= kPersistTokensCap) {
        L.ll_logits = take(t * (E + 1) * 8);
        L.ll_hs = take(t * Is * 8);
        L.ll_h = take(t * K * I * 8);
        L.ll_resid = take(t * H * 8);
    }
    if (T > kLayerDecodeMaxTokens) {
        const size_t nblk = (t + 31) / 32;
        const size_t max_mb = (t * K) / kBM + E + t / kBM + 2;
        L.cnt_blk = take(nblk * E * 4);
        L.base_blk = take(nblk * E * 4);
        L.mblocks = take(max_mb * sizeof(MBlock));
        L.n_mblocks = take(16);
        L.lgp = take(size_t(kRouterSplitMax) * t * (E + 1) * 4);
        L.xg = take((t * K + t) * H * 2);
        L.h16 = take(t * K * I * 2);
        L.hs16 = take(t * Is * 2);
        L.y = take(t * K * H * 2);
        L.ysh = take(t * H * 2);
    }
    L.total = o;
    return L;
}

// Events of moe_layer_profile, per host thread.
struct Prof {
    cudaEvent_t ev[64];
    int n;
};
static thread_local Prof* t_prof = nullptr;

void prof_after_launch(cudaStream_t s) {
    Prof* p = t_prof;
    if (p == nullptr || p->n >= 64) return;
    if (cudaEventCreate(&p->ev[p->n]) != cudaSuccess) return;
    cudaEventRecord(p->ev[p->n], s);
    ++p->n;
}

Dev device_info() {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    int sms = cache[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0)
            sms = 1;
        cache[dev].store(sms, std::memory_order_relaxed);
    }
    return Dev{sms};
}

}  // namespace strata

using namespace strata;

namespace {

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

bool dims_ok(const strata_moe_dims* d) {
    if (d == nullptr) return false;
    if (d->group != 32) return false;
    if (d->hidden < 256 || d->hidden > 4096 || d->hidden % 256 != 0) return false;
    if (d->n_experts < 1 || d->n_experts > kMaxExperts) return false;
    if (d->top_k < 1 || d->top_k > kMaxTopK || d->top_k > d->n_experts) return false;
    if (!pow2_in(d->inter, 64, 1024) || !pow2_in(d->shared_inter, 64, 1024)) return false;
    return true;
}

bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool opt4(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

enum Need { kRouter = 1, kRouted = 2, kShared = 4 };

bool layer_ok(const strata_moe_layer* L, int need) {
    if (L == nullptr) return false;
    if ((need & kRouter) && (!al16(L->router_dev) || !opt4(L->router_bias_dev))) return false;
    if ((need & kRouted) &&
        (!al16(L->gu_q_dev) || !al16(L->gu_s_dev) || !al16(L->dn_q_dev) || !al16(L->dn_s_dev)))
        return false;
    if ((need & kShared) && (!al16(L->sh_gu_q_dev) || !al16(L->sh_gu_s_dev) ||
                             !al16(L->sh_dn_q_dev) || !al16(L->sh_dn_s_dev)))
        return false;
    return true;
}

bool ws_ok(const strata_moe_dims* d, int T, const void* ws, size_t bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return false;
    return bytes >= ws_layout(*d, T).total;
}

template <typename P>
P* at(void* ws, size_t off) {
    return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

// The last CUDA error a call of this host thread met (strata_last_cuda_error).
thread_local cudaError_t t_last_cuda = cudaSuccess;

strata_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return STRATA_OK;
    t_last_cuda = e;
    return STRATA_ECUDA;
}

#define STRATA_TRY(expr)                                   \
    do {                                                   \
        const cudaError_t _e = (expr);                     \
        if (_e != cudaSuccess) return cuda_status(_e);     \
    } while (0)

// The three decode stages.  Stage 1 computes the logits and the shared
// expert's SwiGLU vectors; stage 2 routes (or takes forced ids), buckets,
// publishes the routing and the plan, and runs the routed gate/up; stage 3
// the down products and the combine.
strata_status stage_route(const strata_moe_dims* d, const strata_moe_layer* L, const void* x,
                          int T, bool forced, void* ws, cudaStream_t s) {
    const WsLayout W = ws_layout(*d, T);
    RouteLaunch r{};
    r.router = static_cast<const uint16_t*>(L->router_dev);
    r.bias = L->router_bias_dev;
    r.x = static_cast<const uint16_t*>(x);
    r.logits = at<float>(ws, W.logits);
    r.shq = L->sh_gu_q_dev;
    r.shs = L->sh_gu_s_dev;
    r.hs = at<float>(ws, W.hs);
    r.Is = d->shared_inter;
    r.do_shared = 1;
    r.do_select = forced ? 0 : 1;
    r.T = T;
    r.H = d->hidden;
    r.E = d->n_experts;
    r.K = d->top_k;
    return cuda_status(launch_route_decode(r, s));
}

strata_status stage_gate_up(const strata_moe_dims* d, const strata_moe_layer* L, const void* x,
                            int T, const int32_t* forced_ids, const float* forced_w,
                            int32_t* ids_user, float* w_user, float* sig_user, void* ws,
                            cudaStream_t s, int tail_skip = 0) {
    const WsLayout W = ws_layout(*d, T);
    GuLaunch g{};
    g.q = L->gu_q_dev;
    g.sc = L->gu_s_dev;
    g.x = static_cast<const uint16_t*>(x);
    g.logits = at<float>(ws, W.logits);
    g.forced_ids = forced_ids;
    g.forced_w = forced_w;
    g.ids = at<int32_t>(ws, W.ids);
    g.w = at<float>(ws, W.w);
    g.sig = at<float>(ws, W.sig);
    g.ids_user = ids_user;
    g.w_user = w_user;
    g.sig_user = sig_user;
    g.counts = at<int32_t>(ws, W.counts);
    g.offsets = at<int32_t>(ws, W.offsets);
    g.perm = at<int32_t>(ws, W.perm);
    g.inv = at<int32_t>(ws, W.inv);
    g.plan_out = at<int32_t>(ws, W.plan);
    g.h = at<float>(ws, W.h);
    g.err = &at<Ctl>(ws, W.ctl)->err;
    g.T = T;
    g.H = d->hidden;
    g.I = d->inter;
    g.E = d->n_experts;
    g.K = d->top_k;
    g.mode = kGuRoute;
    g.tail_skip = tail_skip;
    return cuda_status(launch_gate_up_decode(g, s));
}

strata_status stage_down(const strata_moe_dims* d, const strata_moe_layer* L, int T, void* out,
                         float* resid, void* ws, cudaStream_t s) {
    const WsLayout W = ws_layout(*d, T);
    DownLaunch dn{};
    dn.q = L->dn_q_dev;
    dn.sc = L->dn_s_dev;
    dn.shq = L->sh_dn_q_dev;
    dn.shs = L->sh_dn_s_dev;
    dn.h = at<float>(ws, W.h);
    dn.hs = at<float>(ws, W.hs);
    dn.plan = at<int32_t>(ws, W.plan);
    dn.inv = at<int32_t>(ws, W.inv);
    dn.w = at<float>(ws, W.w);
    dn.sig = at<float>(ws, W.sig);
    dn.out = static_cast<uint16_t*>(out);
    dn.resid = resid;
    dn.err = &at<Ctl>(ws, W.ctl)->err;
    dn.T = T;
    dn.H = d->hidden;
    dn.I = d->inter;
    dn.Is = d->shared_inter;
    dn.E = d->n_experts;
    dn.K = d->top_k;
    dn.mode = kDownFused;
    return cuda_status(launch_down_decode(dn, s));
}

// One layer on the decode kernels.  forced_ids/forced_w: NULL to route.
// resid: NULL, or the residual that gets += the bf16 output.  tail_skip: 0,
// or the place past which an expert every token ranks there is left out.
strata_status decode_layer(const strata_moe_dims* d, const strata_moe_layer* L, const void* x,
                           int T, const int32_t* forced_ids, const float* forced_w,
                           int32_t* ids_user, float* w_user, float* sig_user, void* out,
                           float* resid, void* ws, cudaStream_t s, int tail_skip = 0) {
    strata_status st = stage_route(d, L, x, T, forced_ids != nullptr, ws, s);
    if (st != STRATA_OK) return st;
    st = stage_gate_up(d, L, x, T, forced_ids, forced_w, ids_user, w_user, sig_user, ws, s,
                       tail_skip);
    if (st != STRATA_OK) return st;
    return stage_down(d, L, T, out, resid, ws, s);
}

// One layer on the prefill (tcgen05) kernels.
strata_status prefill_layer(const strata_moe_dims* d, const strata_moe_layer* L, const void* x,
                            int T, const int32_t* forced_ids, const float* forced_w,
                            int32_t* ids_user, float* w_user, float* sig_user, void* out,
                            float* resid, void* ws, cudaStream_t s) {
    if (!prefill_supported(*d)) return STRATA_EUNSUPPORTED;
    const WsLayout W = ws_layout(*d, T);
    uint32_t* err = &at<Ctl>(ws, W.ctl)->err;
    PfRoute r{};
    r.x = static_cast<const uint16_t*>(x);
    r.router = static_cast<const uint16_t*>(L->router_dev);
    r.part = at<float>(ws, W.lgp);
    r.forced_ids = forced_ids;
    r.forced_w = forced_w;
    r.ids = at<int32_t>(ws, W.ids);
    r.w = at<float>(ws, W.w);
    r.sig = at<float>(ws, W.sig);
    r.ids_user = ids_user;
    r.w_user = w_user;
    r.sig_user = sig_user;
    r.err = err;
    r.T = T;
    r.H = d->hidden;
    r.E = d->n_experts;
    r.K = d->top_k;
    r.bias = L->router_bias_dev;
    STRATA_TRY(launch_prefill_route(r, s));
    PfBucket b{};
    b.ids = r.ids;
    b.cnt_blk = at<int32_t>(ws, W.cnt_blk);
    b.base_blk = at<int32_t>(ws, W.base_blk);
    b.counts = at<int32_t>(ws, W.counts);
    b.offsets = at<int32_t>(ws, W.offsets);
    b.perm = at<int32_t>(ws, W.perm);
    b.inv = at<int32_t>(ws, W.inv);
    b.mblocks = at<MBlock>(ws, W.mblocks);
    b.n_mblocks = at<int32_t>(ws, W.n_mblocks);
    b.err = err;
    b.T = T;
    b.K = d->top_k;
    b.E = d->n_experts;
    b.with_shared = 1;
    STRATA_TRY(launch_prefill_bucket(b, s));
    PfExperts p{};
    p.x = r.x;
    p.perm = b.perm;
    p.xg = at<__half>(ws, W.xg);
    p.gu_q = L->gu_q_dev;
    p.gu_s = L->gu_s_dev;
    p.dn_q = L->dn_q_dev;
    p.dn_s = L->dn_s_dev;
    p.sh_gu_q = L->sh_gu_q_dev;
    p.sh_gu_s = L->sh_gu_s_dev;
    p.sh_dn_q = L->sh_dn_q_dev;
    p.sh_dn_s = L->sh_dn_s_dev;
    p.mblocks = b.mblocks;
    p.n_mblocks = b.n_mblocks;
    p.h = at<__half>(ws, W.h16);
    p.hs = at<__half>(ws, W.hs16);
    p.y = at<__half>(ws, W.y);
    p.ysh = at<__half>(ws, W.ysh);
    p.err = err;
    p.T = T;
    p.K = d->top_k;
    p.H = d->hidden;
    p.I = d->inter;
    p.Is = d->shared_inter;
    p.E = d->n_experts;
    p.routed = 1;
    p.shared = 1;
    p.xg_rows = T * d->top_k + T;
    p.xg_shared_row0 = T * d->top_k;
    STRATA_TRY(launch_prefill_experts(p, s));
    STRATA_TRY(launch_prefill_combine(p.y, nullptr, p.ysh, b.inv, r.w, r.sig, T, d->top_k,
                                      d->hidden, static_cast<uint16_t*>(out), resid, p.err, s));
    return STRATA_OK;
}

// Prefill operands of a stage-wise call at T > kDecodeMaxTokens: the
// workspace's block list, fp16 operands and shared-expert outputs.
PfExperts pf_stage(const strata_moe_dims* d, const strata_moe_layer* L, int T, void* ws) {
    const WsLayout W = ws_layout(*d, T);
    PfExperts p{};
    p.gu_q = L->gu_q_dev;
    p.gu_s = L->gu_s_dev;
    p.dn_q = L->dn_q_dev;
    p.dn_s = L->dn_s_dev;
    p.sh_gu_q = L->sh_gu_q_dev;
    p.sh_gu_s = L->sh_gu_s_dev;
    p.sh_dn_q = L->sh_dn_q_dev;
    p.sh_dn_s = L->sh_dn_s_dev;
    p.xg = at<__half>(ws, W.xg);
    p.mblocks = at<MBlock>(ws, W.mblocks);
    p.n_mblocks = at<int32_t>(ws, W.n_mblocks);
    p.h = at<__half>(ws, W.h16);
    p.hs = at<__half>(ws, W.hs16);
    p.y = at<__half>(ws, W.y);
    p.ysh = at<__half>(ws, W.ysh);
    p.err = &at<Ctl>(ws, W.ctl)->err;
    p.T = T;
    p.K = d->top_k;
    p.H = d->hidden;
    p.I = d->inter;
    p.Is = d->shared_inter;
    p.E = d->n_experts;
    return p;
}

// Routed gate/up at T > kDecodeMaxTokens from caller offsets/perm: block
// list, gather, GEMM.  h_f32: NULL to keep h only as the fp16 operand.
strata_status pf_gate_up(const strata_moe_dims* d, const strata_moe_layer* L, const void* x,
                         int T, const int32_t* offsets, const int32_t* perm, float* h_f32,
                         void* ws, cudaStream_t s) {
    if (!prefill_supported(*d)) return STRATA_EUNSUPPORTED;
    PfExperts p = pf_stage(d, L, T, ws);
    p.x = static_cast<const uint16_t*>(x);
    p.perm = perm;
    p.routed = 1;
    p.xg_rows = T * d->top_k;
    p.h_f32 = h_f32;
    STRATA_TRY(launch_prefill_blocks(offsets, T, d->top_k, d->n_experts, 0,
                                     const_cast<MBlock*>(p.mblocks),
                                     const_cast<int32_t*>(p.n_mblocks), p.err, s));
    STRATA_TRY(launch_prefill_gather(p.x, perm, T, d->top_k, d->hidden, p.xg, p.xg_rows, p.err,
                                     s));
    STRATA_TRY(launch_prefill_gate_up(p, s));
    return STRATA_OK;
}

// Routed down at T > kDecodeMaxTokens into bf16 y (slot order); A is the
// workspace's fp16 h, the block list the one pf_gate_up or the caller's
// offsets built.
strata_status pf_down(const strata_moe_dims* d, const strata_moe_layer* L, int T,
                      const int32_t* offsets, bool build_blocks, void* y, void* ws,
                      cudaStream_t s) {
    if (!prefill_supported(*d)) return STRATA_EUNSUPPORTED;
    PfExperts p = pf_stage(d, L, T, ws);
    p.routed = 1;
    p.y_bf16 = static_cast<uint16_t*>(y);
    if (build_blocks)
        STRATA_TRY(launch_prefill_blocks(offsets, T, d->top_k, d->n_experts, 0,
                                         const_cast<MBlock*>(p.mblocks),
                                         const_cast<int32_t*>(p.n_mblocks), p.err, s));
    STRATA_TRY(launch_prefill_down(p, s));
    return STRATA_OK;
}

// n_layers residual layers (resid != NULL) or one layer on x_in, as
// persistent-kernel launches of up to kPxMaxLayers layers each;
// STRATA_EUNSUPPORTED (nothing launched) when that kernel does not take the
// shape or T.
strata_status persist_layers(const strata_moe_dims* d, const strata_moe_layer* layers,
                             int n_layers, const void* x_in, float* resid, float eps, int T,
                             const int32_t* forced_ids, const float* forced_w, int32_t* ids_user,
                             float* w_user, float* sig_user, void* out, void* x_out, void* ws,
                             cudaStream_t s) {
    PxGeo g;
    if ((x_in == nullptr) == (resid == nullptr) || (x_in != nullptr && n_layers != 1) ||
        !px_geometry(*d, T, forced_ids != nullptr, resid != nullptr, device_info().sms, &g))
        return STRATA_EUNSUPPORTED;
    const WsLayout W = ws_layout(*d, T);
    PxArgs a{};
    a.T = T;
    a.H = d->hidden;
    a.E = d->n_experts;
    a.K = d->top_k;
    a.I = d->inter;
    a.Is = d->shared_inter;
    a.eps = eps;
    a.x_in = static_cast<const uint16_t*>(x_in);
    a.resid = resid;
    a.ll_logits = at<uint64_t>(ws, W.ll_logits);
    a.ll_hs = at<uint64_t>(ws, W.ll_hs);
    a.ll_h = at<uint64_t>(ws, W.ll_h);
    a.ll_resid = at<uint64_t>(ws, W.ll_resid);
    a.ids = at<int32_t>(ws, W.ids);
    a.w = at<float>(ws, W.w);
    a.sig = at<float>(ws, W.sig);
    a.counts = at<int32_t>(ws, W.counts);
    a.offsets = at<int32_t>(ws, W.offsets);
    a.perm = at<int32_t>(ws, W.perm);
    a.inv = at<int32_t>(ws, W.inv);
    a.flags = at<uint32_t>(ws, W.flags);
    a.err = &at<Ctl>(ws, W.ctl)->err;
    a.grid_wait_limit = grid_wait_limit();
    a.R = g.R;
    a.gu_stages = g.gu_stages;
    a.dn_stages = g.dn_stages;
    a.off_x = g.off_x;
    a.off_r = g.off_r;
    a.off_sd = g.off_sd;
    a.off_d = g.off_d;
    a.off_y = g.off_y;
    a.off_g = g.off_g;
    a.sd_q = g.sd_q;
    a.sd_bytes = g.sd_bytes;
    a.d_q = g.d_q;
    a.d_stage = g.d_stage;
    a.g_q = g.g_q;
    a.g_stage = g.g_stage;
    const size_t TK = size_t(T) * d->top_k;
    for (int c0 = 0; c0 < n_layers; c0 += kPxMaxLayers) {
        const int n = n_layers - c0 < kPxMaxLayers ? n_layers - c0 : kPxMaxLayers;
        const bool last = c0 + n == n_layers;
        a.n_layers = n;
        for (int l = 0; l < n; ++l) {
            const strata_moe_layer& L = layers[c0 + l];
            a.L[l] = PxLayer{static_cast<const uint16_t*>(L.router_dev), L.router_bias_dev,
                             L.gu_q_dev, L.gu_s_dev, L.dn_q_dev, L.dn_s_dev,
                             L.sh_gu_q_dev, L.sh_gu_s_dev, L.sh_dn_q_dev, L.sh_dn_s_dev};
        }
        a.forced_ids = forced_ids ? forced_ids + size_t(c0) * TK : nullptr;
        a.forced_w = forced_w ? forced_w + size_t(c0) * TK : nullptr;
        a.out = last ? static_cast<uint16_t*>(out) : nullptr;
        a.x_out = last ? static_cast<uint16_t*>(x_out) : nullptr;
        a.ids_user = last ? ids_user : nullptr;
        a.w_user = last ? w_user : nullptr;
        a.sig_user = last ? sig_user : nullptr;
        STRATA_TRY(launch_persistent(a, g, s));
    }
    return STRATA_OK;
}

// The layer at any T: the persistent decode kernel where it takes the shape
// and T, else the three decode kernels up to kLayerDecodeMaxTokens (or up to
// kDecodeMaxTokens when the shape does not allow the tensor-core kernels),
// the tensor-core (prefill) kernels above.
strata_status any_layer(const strata_moe_dims* d, const strata_moe_layer* L, const void* x, int T,
                        const int32_t* forced_ids, const float* forced_w, int32_t* ids_user,
                        float* w_user, float* sig_user, void* out, float* resid, void* ws,
                        cudaStream_t s) {
    if (resid == nullptr) {
        const strata_status st = persist_layers(d, L, 1, x, nullptr, 0.0f, T, forced_ids,
                                                forced_w, ids_user, w_user, sig_user, out,
                                                nullptr, ws, s);
        if (st != STRATA_EUNSUPPORTED) return st;
    }
    if (T <= kLayerDecodeMaxTokens || (T <= kDecodeMaxTokens && !prefill_supported(*d)))
        return decode_layer(d, L, x, T, forced_ids, forced_w, ids_user, w_user, sig_user, out,
                            resid, ws, s);
    return prefill_layer(d, L, x, T, forced_ids, forced_w, ids_user, w_user, sig_user, out, resid,
                         ws, s);
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const strata_moe_dims* dims, int32_t max_tokens) {
    if (!dims_ok(dims) || max_tokens < 1) return 0;
    // a call with T <= max_tokens takes the persistent, the decode or the
    // prefill layout; each grows with T
    const int pmax = max_tokens < kPersistTokensCap ? max_tokens : kPersistTokensCap;
    const int dmax = max_tokens < kDecodeMaxTokens ? max_tokens : kDecodeMaxTokens;
    size_t n = ws_layout(*dims, pmax).total;
    const size_t a = ws_layout(*dims, dmax).total, b = ws_layout(*dims, max_tokens).total;
    if (a > n) n = a;
    if (b > n) n = b;
    return n;
}

int32_t moe_decode_max_tokens(void) { return kDecodeMaxTokens; }

int32_t moe_layer_decode_max_tokens(void) { return kLayerDecodeMaxTokens; }

strata_status moe_rmsnorm(const float* r_dev, int32_t T, int32_t H, float eps, void* x_dev,
                          void* stream) {
    if (T < 0 || H < 256 || H > 4096 || H % 256 != 0 || !(eps >= 0.0f)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(r_dev) || !al16(x_dev)) return STRATA_EINVAL;
    return cuda_status(launch_rmsnorm(r_dev, T, H, eps, static_cast<uint16_t*>(x_dev),
                                      static_cast<cudaStream_t>(stream)));
}

strata_status moe_route(const strata_moe_dims* dims, const strata_moe_layer* layer,
                        const void* x_dev, int32_t T, int32_t* ids_dev, float* weights_dev,
                        float* shared_gate_dev, float* logits_dev, void* ws_dev,
                        size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouter)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(x_dev) || !al4(ids_dev) || !al4(weights_dev) || !al4(shared_gate_dev) ||
        !opt4(logits_dev) || !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    const WsLayout W = ws_layout(*dims, T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > kDecodeMaxTokens) {
        if (!prefill_supported(*dims)) return STRATA_EUNSUPPORTED;
        PfRoute r{};
        r.x = static_cast<const uint16_t*>(x_dev);
        r.router = static_cast<const uint16_t*>(layer->router_dev);
        r.bias = layer->router_bias_dev;
        r.part = at<float>(ws_dev, W.lgp);
        r.logits_user = logits_dev;
        r.ids = at<int32_t>(ws_dev, W.ids);
        r.w = at<float>(ws_dev, W.w);
        r.sig = at<float>(ws_dev, W.sig);
        r.ids_user = ids_dev;
        r.w_user = weights_dev;
        r.sig_user = shared_gate_dev;
        r.err = &at<Ctl>(ws_dev, W.ctl)->err;
        r.T = T;
        r.H = dims->hidden;
        r.E = dims->n_experts;
        r.K = dims->top_k;
        return cuda_status(launch_prefill_route(r, s));
    }
    RouteLaunch r{};
    r.router = static_cast<const uint16_t*>(layer->router_dev);
    r.bias = layer->router_bias_dev;
    r.x = static_cast<const uint16_t*>(x_dev);
    r.logits = at<float>(ws_dev, W.logits);
    r.do_shared = 0;
    r.do_select = 1;
    r.T = T;
    r.H = dims->hidden;
    r.E = dims->n_experts;
    r.K = dims->top_k;
    r.Is = dims->shared_inter;
    STRATA_TRY(launch_route_decode(r, s));
    SelectLaunch sl{};
    sl.logits = r.logits;
    sl.ids = ids_dev;
    sl.w = weights_dev;
    sl.sig = shared_gate_dev;
    sl.logits_out = logits_dev;
    sl.err = &at<Ctl>(ws_dev, W.ctl)->err;
    sl.T = T;
    sl.E = dims->n_experts;
    sl.K = dims->top_k;
    return cuda_status(launch_select(sl, s));
}

strata_status moe_permute(const strata_moe_dims* dims, const int32_t* ids_dev, int32_t T,
                          int32_t* counts_dev, int32_t* offsets_dev, int32_t* perm_dev,
                          int32_t* inv_perm_dev, void* ws_dev, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al4(ids_dev) || !al4(counts_dev) || !al4(offsets_dev) || !al4(perm_dev) ||
        !al4(inv_perm_dev) || !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    const WsLayout W = ws_layout(*dims, T);
    if (T > kDecodeMaxTokens) {
        PfBucket b{};
        b.ids = ids_dev;
        b.cnt_blk = at<int32_t>(ws_dev, W.cnt_blk);
        b.base_blk = at<int32_t>(ws_dev, W.base_blk);
        b.counts = counts_dev;
        b.offsets = offsets_dev;
        b.perm = perm_dev;
        b.inv = inv_perm_dev;
        b.mblocks = at<MBlock>(ws_dev, W.mblocks);
        b.n_mblocks = at<int32_t>(ws_dev, W.n_mblocks);
        b.err = &at<Ctl>(ws_dev, W.ctl)->err;
        b.T = T;
        b.K = dims->top_k;
        b.E = dims->n_experts;
        b.with_shared = 0;
        return cuda_status(launch_prefill_bucket(b, static_cast<cudaStream_t>(stream)));
    }
    return cuda_status(launch_permute_small(ids_dev, T, dims->top_k, dims->n_experts, counts_dev,
                                            offsets_dev, perm_dev, inv_perm_dev,
                                            &at<Ctl>(ws_dev, W.ctl)->err,
                                            static_cast<cudaStream_t>(stream)));
}

strata_status moe_expert_gate_up(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                 const void* x_dev, int32_t T, const int32_t* offsets_dev,
                                 const int32_t* perm_dev, float* h_dev, void* ws_dev,
                                 size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouted)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(x_dev) || !al4(offsets_dev) || !al4(perm_dev) || !al16(h_dev) ||
        !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > kDecodeMaxTokens)
        return pf_gate_up(dims, layer, x_dev, T, offsets_dev, perm_dev, h_dev, ws_dev, s);
    const WsLayout W = ws_layout(*dims, T);
    int32_t* plan = at<int32_t>(ws_dev, W.plan);
    STRATA_TRY(launch_plan(offsets_dev, perm_dev, T, dims->top_k, dims->n_experts, plan,
                           &at<Ctl>(ws_dev, W.ctl)->err, s));
    GuLaunch g{};
    g.q = layer->gu_q_dev;
    g.sc = layer->gu_s_dev;
    g.x = static_cast<const uint16_t*>(x_dev);
    g.plan = plan;
    g.h = h_dev;
    g.err = &at<Ctl>(ws_dev, W.ctl)->err;
    g.T = T;
    g.H = dims->hidden;
    g.I = dims->inter;
    g.E = dims->n_experts;
    g.K = dims->top_k;
    g.mode = kGuPlan;
    return cuda_status(launch_gate_up_decode(g, s));
}

strata_status moe_expert_down(const strata_moe_dims* dims, const strata_moe_layer* layer,
                              const float* h_dev, int32_t T, const int32_t* offsets_dev,
                              void* y_dev, void* ws_dev, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouted)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(h_dev) || !al4(offsets_dev) || !al16(y_dev) || !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > kDecodeMaxTokens) {
        if (!prefill_supported(*dims)) return STRATA_EUNSUPPORTED;
        const WsLayout W = ws_layout(*dims, T);
        STRATA_TRY(launch_prefill_pack(h_dev, (long long)T * dims->top_k * dims->inter,
                                       at<__half>(ws_dev, W.h16), &at<Ctl>(ws_dev, W.ctl)->err,
                                       s));
        return pf_down(dims, layer, T, offsets_dev, true, y_dev, ws_dev, s);
    }
    const WsLayout W = ws_layout(*dims, T);
    int32_t* plan = at<int32_t>(ws_dev, W.plan);
    STRATA_TRY(launch_plan(offsets_dev, nullptr, T, dims->top_k, dims->n_experts, plan,
                           &at<Ctl>(ws_dev, W.ctl)->err, s));
    DownLaunch dn{};
    dn.q = layer->dn_q_dev;
    dn.sc = layer->dn_s_dev;
    dn.h = h_dev;
    dn.plan = plan;
    dn.y_out = static_cast<uint16_t*>(y_dev);
    dn.err = &at<Ctl>(ws_dev, W.ctl)->err;
    dn.T = T;
    dn.H = dims->hidden;
    dn.I = dims->inter;
    dn.Is = dims->shared_inter;
    dn.E = dims->n_experts;
    dn.K = dims->top_k;
    dn.mode = kDownSlots;
    return cuda_status(launch_down_decode(dn, s));
}

strata_status moe_expert_ffn(const strata_moe_dims* dims, const strata_moe_layer* layer,
                             const void* x_dev, int32_t T, const int32_t* offsets_dev,
                             const int32_t* perm_dev, void* y_dev, void* ws_dev,
                             size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouted)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(x_dev) || !al4(offsets_dev) || !al4(perm_dev) || !al16(y_dev) ||
        !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    if (T > kDecodeMaxTokens) {
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        const strata_status st =
            pf_gate_up(dims, layer, x_dev, T, offsets_dev, perm_dev, nullptr, ws_dev, s);
        if (st != STRATA_OK) return st;
        return pf_down(dims, layer, T, offsets_dev, false, y_dev, ws_dev, s);
    }
    const WsLayout W = ws_layout(*dims, T);
    float* h = at<float>(ws_dev, W.h);
    strata_status st = moe_expert_gate_up(dims, layer, x_dev, T, offsets_dev, perm_dev, h,
                                          ws_dev, ws_bytes, stream);
    if (st != STRATA_OK) return st;
    return moe_expert_down(dims, layer, h, T, offsets_dev, y_dev, ws_dev, ws_bytes, stream);
}

strata_status moe_combine(const strata_moe_dims* dims, const strata_moe_layer* layer,
                          const void* x_dev, int32_t T, const void* y_dev,
                          const int32_t* inv_perm_dev, const float* weights_dev,
                          const float* shared_gate_dev, void* out_dev, void* ws_dev,
                          size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kShared)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(x_dev) || !al16(y_dev) || !al4(inv_perm_dev) || !al4(weights_dev) ||
        !al4(shared_gate_dev) || !al16(out_dev) || !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    const WsLayout W = ws_layout(*dims, T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > kDecodeMaxTokens) {
        // the shared expert over the T tokens, then the combine of bf16 y
        if (!prefill_supported(*dims)) return STRATA_EUNSUPPORTED;
        PfExperts p = pf_stage(dims, layer, T, ws_dev);
        p.x = static_cast<const uint16_t*>(x_dev);
        p.shared = 1;
        p.xg_rows = T;
        p.xg_shared_row0 = 0;
        STRATA_TRY(launch_prefill_blocks(nullptr, T, dims->top_k, dims->n_experts, 1,
                                         const_cast<MBlock*>(p.mblocks),
                                         const_cast<int32_t*>(p.n_mblocks), p.err, s));
        STRATA_TRY(launch_prefill_gather(p.x, nullptr, T, 0, dims->hidden, p.xg, T, p.err, s));
        STRATA_TRY(launch_prefill_gate_up(p, s));
        STRATA_TRY(launch_prefill_down(p, s));
        STRATA_TRY(launch_prefill_combine(nullptr, static_cast<const uint16_t*>(y_dev), p.ysh,
                                          inv_perm_dev, weights_dev, shared_gate_dev, T,
                                          dims->top_k, dims->hidden,
                                          static_cast<uint16_t*>(out_dev), nullptr, p.err, s));
        return STRATA_OK;
    }
    GuLaunch g{};
    g.q = layer->sh_gu_q_dev;
    g.sc = layer->sh_gu_s_dev;
    g.x = static_cast<const uint16_t*>(x_dev);
    g.h = at<float>(ws_dev, W.hs);
    g.err = &at<Ctl>(ws_dev, W.ctl)->err;
    g.T = T;
    g.H = dims->hidden;
    g.I = dims->shared_inter;
    g.E = 1;
    g.K = 1;
    g.mode = kGuShared;
    STRATA_TRY(launch_gate_up_decode(g, s));
    DownLaunch dn{};
    dn.shq = layer->sh_dn_q_dev;
    dn.shs = layer->sh_dn_s_dev;
    dn.hs = g.h;
    dn.inv = inv_perm_dev;
    dn.w = weights_dev;
    dn.sig = shared_gate_dev;
    dn.y_in = static_cast<const uint16_t*>(y_dev);
    dn.out = static_cast<uint16_t*>(out_dev);
    dn.err = g.err;
    dn.T = T;
    dn.H = dims->hidden;
    dn.I = dims->inter;
    dn.Is = dims->shared_inter;
    dn.E = dims->n_experts;
    dn.K = dims->top_k;
    dn.mode = kDownCombine;
    return cuda_status(launch_down_decode(dn, s));
}

strata_status moe_layer_forward(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                const void* x_dev, int32_t T, int32_t* ids_dev,
                                float* weights_dev, float* shared_gate_dev, void* out_dev,
                                void* ws_dev, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouter | kRouted | kShared))
        return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(x_dev) || !opt4(ids_dev) || !opt4(weights_dev) || !opt4(shared_gate_dev) ||
        !al16(out_dev) || !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    return any_layer(dims, layer, x_dev, T, nullptr, nullptr, ids_dev, weights_dev,
                     shared_gate_dev, out_dev, nullptr, ws_dev, static_cast<cudaStream_t>(stream));
}

strata_status moe_layer_forward_routed(const strata_moe_dims* dims,
                                       const strata_moe_layer* layer, const void* x_dev,
                                       int32_t T, const int32_t* ids_dev,
                                       const float* weights_dev, void* out_dev, void* ws_dev,
                                       size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouter | kRouted | kShared))
        return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(x_dev) || !al4(ids_dev) || !al4(weights_dev) || !al16(out_dev) ||
        !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    return any_layer(dims, layer, x_dev, T, ids_dev, weights_dev, nullptr, nullptr, nullptr,
                     out_dev, nullptr, ws_dev, static_cast<cudaStream_t>(stream));
}

strata_status moe_layer_forward_tail_skip(const strata_moe_dims* dims,
                                          const strata_moe_layer* layer, const void* x_dev,
                                          int32_t T, int32_t tail_skip,
                                          const int32_t* forced_ids_dev,
                                          const float* forced_weights_dev, int32_t* ids_dev,
                                          float* weights_dev, float* shared_gate_dev,
                                          void* out_dev, void* ws_dev, size_t ws_bytes,
                                          void* stream) {
    if (!dims_ok(dims) || T < 0 || tail_skip < 0 ||
        !layer_ok(layer, kRouter | kRouted | kShared) ||
        ((forced_ids_dev == nullptr) != (forced_weights_dev == nullptr)))
        return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(x_dev) || !opt4(forced_ids_dev) || !opt4(forced_weights_dev) || !opt4(ids_dev) ||
        !opt4(weights_dev) || !opt4(shared_gate_dev) || !al16(out_dev) ||
        !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // a decode window: the decode kernels with the skip; a prompt batch is
    // not touched
    if (T <= kDecodeMaxTokens)
        return decode_layer(dims, layer, x_dev, T, forced_ids_dev, forced_weights_dev, ids_dev,
                            weights_dev, shared_gate_dev, out_dev, nullptr, ws_dev, s,
                            tail_skip < dims->top_k ? tail_skip : 0);
    return any_layer(dims, layer, x_dev, T, forced_ids_dev, forced_weights_dev, ids_dev,
                     weights_dev, shared_gate_dev, out_dev, nullptr, ws_dev, s);
}

strata_status moe_block_forward(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                float* resid_dev, int32_t T, float eps, const int32_t* ids_dev,
                                const float* weights_dev, void* x_out_dev, void* out_dev,
                                void* ws_dev, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouter | kRouted | kShared) ||
        !(eps >= 0.0f))
        return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(resid_dev) || (ids_dev == nullptr) != (weights_dev == nullptr) ||
        !opt4(ids_dev) || !opt4(weights_dev) ||
        (x_out_dev && !al16(x_out_dev)) || (out_dev && !al16(out_dev)) ||
        !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    const WsLayout W = ws_layout(*dims, T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const strata_status st = persist_layers(dims, layer, 1, nullptr, resid_dev, eps, T, ids_dev,
                                            weights_dev, nullptr, nullptr, nullptr, out_dev,
                                            x_out_dev, ws_dev, s);
    if (st != STRATA_EUNSUPPORTED) return st;
    void* x = x_out_dev ? x_out_dev : at<void>(ws_dev, W.x);
    void* out = out_dev ? out_dev : at<void>(ws_dev, W.out);
    STRATA_TRY(launch_rmsnorm(resid_dev, T, dims->hidden, eps, static_cast<uint16_t*>(x), s));
    return any_layer(dims, layer, x, T, ids_dev, weights_dev, nullptr, nullptr, nullptr, out,
                     resid_dev, ws_dev, s);
}

strata_status moe_stack_forward(const strata_moe_dims* dims, const strata_moe_layer* layers,
                                int32_t n_layers, float* resid_dev, int32_t T, float eps,
                                const int32_t* ids_dev, const float* weights_dev, void* out_dev,
                                void* ws_dev, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || n_layers < 0 || layers == nullptr || !(eps >= 0.0f))
        return STRATA_EINVAL;
    for (int l = 0; l < n_layers; ++l)
        if (!layer_ok(layers + l, kRouter | kRouted | kShared)) return STRATA_EINVAL;
    if (T == 0 || n_layers == 0) return STRATA_OK;
    if (!al16(resid_dev) || (out_dev && !al16(out_dev)) ||
        (ids_dev == nullptr) != (weights_dev == nullptr) || !opt4(ids_dev) ||
        !opt4(weights_dev) || !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    const size_t TK = size_t(T) * dims->top_k;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const strata_status pst = persist_layers(dims, layers, n_layers, nullptr, resid_dev, eps, T,
                                             ids_dev, weights_dev, nullptr, nullptr, nullptr,
                                             out_dev, nullptr, ws_dev, s);
    if (pst != STRATA_EUNSUPPORTED) return pst;
    for (int l = 0; l < n_layers; ++l) {
        const strata_status st = moe_block_forward(
            dims, layers + l, resid_dev, T, eps, ids_dev ? ids_dev + l * TK : nullptr,
            weights_dev ? weights_dev + l * TK : nullptr, nullptr,
            l + 1 == n_layers ? out_dev : nullptr, ws_dev, ws_bytes, stream);
        if (st != STRATA_OK) return st;
    }
    return STRATA_OK;
}

strata_status moe_decode_route(const strata_moe_dims* dims, const strata_moe_layer* layer,
                               const void* x_dev, int32_t T, int32_t forced, void* ws_dev,
                               size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouter | kShared)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (T > kDecodeMaxTokens || !al16(x_dev) || !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    return stage_route(dims, layer, x_dev, T, forced != 0, ws_dev,
                       static_cast<cudaStream_t>(stream));
}

strata_status moe_decode_gate_up(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                 const void* x_dev, int32_t T, const int32_t* forced_ids_dev,
                                 const float* forced_weights_dev, int32_t* ids_dev,
                                 float* weights_dev, float* shared_gate_dev, void* ws_dev,
                                 size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouted)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (T > kDecodeMaxTokens || !al16(x_dev) ||
        (forced_ids_dev == nullptr) != (forced_weights_dev == nullptr) ||
        !opt4(forced_ids_dev) || !opt4(forced_weights_dev) || !opt4(ids_dev) ||
        !opt4(weights_dev) || !opt4(shared_gate_dev) || !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    return stage_gate_up(dims, layer, x_dev, T, forced_ids_dev, forced_weights_dev, ids_dev,
                         weights_dev, shared_gate_dev, ws_dev, static_cast<cudaStream_t>(stream));
}

strata_status moe_decode_down_combine(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                      int32_t T, void* out_dev, float* resid_dev, void* ws_dev,
                                      size_t ws_bytes, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouted | kShared)) return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (T > kDecodeMaxTokens || !al16(out_dev) || (resid_dev && !al16(resid_dev)) ||
        !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    return stage_down(dims, layer, T, out_dev, resid_dev, ws_dev,
                      static_cast<cudaStream_t>(stream));
}


strata_status moe_layer_profile(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                const void* x_dev, int32_t T, void* out_dev, void* ws_dev,
                                size_t ws_bytes, void* stream, float* us, int32_t max_n,
                                int32_t* n_out) {
    if (!dims_ok(dims) || T < 1 || !layer_ok(layer, kRouter | kRouted | kShared) ||
        !al16(x_dev) || !al16(out_dev) || us == nullptr || n_out == nullptr || max_n < 1 ||
        !ws_ok(dims, T, ws_dev, ws_bytes))
        return STRATA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Prof prof{};
    cudaEvent_t start;
    if (cudaEventCreate(&start) != cudaSuccess) return STRATA_ECUDA;
    cudaEventRecord(start, s);
    t_prof = &prof;
    const strata_status st = any_layer(dims, layer, x_dev, T, nullptr, nullptr, nullptr, nullptr,
                                       nullptr, out_dev, nullptr, ws_dev, s);
    t_prof = nullptr;
    strata_status rc = st;
    if (cudaStreamSynchronize(s) != cudaSuccess) rc = STRATA_ECUDA;
    int n = 0;
    cudaEvent_t prev = start;
    for (int i = 0; i < prof.n; ++i) {
        float ms = 0.0f;
        if (rc == STRATA_OK && cudaEventElapsedTime(&ms, prev, prof.ev[i]) != cudaSuccess)
            rc = STRATA_ECUDA;
        if (n < max_n) us[n++] = ms * 1000.0f;
        prev = prof.ev[i];
    }
    const int total = prof.n;
    for (int i = 0; i < prof.n; ++i) cudaEventDestroy(prof.ev[i]);
    cudaEventDestroy(start);
    *n_out = total;
    return rc;
}

strata_status moe_get_device_status(void* ws_dev, void* stream) {
    if (ws_dev == nullptr || (reinterpret_cast<uintptr_t>(ws_dev) & 255u) != 0)
        return STRATA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    Ctl* ctl = static_cast<Ctl*>(ws_dev);
    if (cudaMemcpyAsync(&word, &ctl->err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return STRATA_ECUDA;
    if (cudaMemsetAsync(&ctl->err, 0, sizeof(uint32_t), s) != cudaSuccess) return STRATA_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return STRATA_ECUDA;
    return static_cast<strata_status>(word);
}

int32_t moe_layer_path(const strata_moe_dims* dims, int32_t T, int32_t forced) {
    if (!dims_ok(dims) || T < 1) return 0;
    PxGeo g;
    if (px_geometry(*dims, T, forced != 0, false, device_info().sms, &g))
        return STRATA_PATH_PERSISTENT;
    if (T <= kLayerDecodeMaxTokens || (T <= kDecodeMaxTokens && !prefill_supported(*dims)))
        return STRATA_PATH_DECODE;
    return prefill_supported(*dims) ? STRATA_PATH_TC : 0;
}

strata_status moe_layer_bucketing(const strata_moe_dims* dims, int32_t T, const void* ws_dev,
                                  size_t ws_bytes, int32_t* counts_dev, int32_t* offsets_dev,
                                  int32_t* perm_dev, int32_t* inv_dev, void* stream) {
    if (!dims_ok(dims) || T < 1 || !ws_ok(dims, T, ws_dev, ws_bytes) || !al4(counts_dev) ||
        !al4(offsets_dev) || !al4(perm_dev) || !al4(inv_dev))
        return STRATA_EINVAL;
    const WsLayout W = ws_layout(*dims, T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* w = const_cast<void*>(ws_dev);
    const size_t E = size_t(dims->n_experts), TK = size_t(T) * dims->top_k;
    STRATA_TRY(cudaMemcpyAsync(counts_dev, at<int32_t>(w, W.counts), E * 4,
                               cudaMemcpyDeviceToDevice, s));
    STRATA_TRY(cudaMemcpyAsync(offsets_dev, at<int32_t>(w, W.offsets), (E + 1) * 4,
                               cudaMemcpyDeviceToDevice, s));
    STRATA_TRY(cudaMemcpyAsync(perm_dev, at<int32_t>(w, W.perm), TK * 4,
                               cudaMemcpyDeviceToDevice, s));
    STRATA_TRY(cudaMemcpyAsync(inv_dev, at<int32_t>(w, W.inv), TK * 4,
                               cudaMemcpyDeviceToDevice, s));
    return STRATA_OK;
}

void strata_set_grid_wait_limit(uint32_t polls) { set_grid_wait_limit(polls); }

strata_status strata_px_trace_read(void* host, size_t bytes) {
    if (host == nullptr || bytes == 0) return STRATA_EINVAL;
    const cudaError_t e = px_trace_copy(host, bytes);
    if (e == cudaErrorNotSupported) return STRATA_EUNSUPPORTED;
    return cuda_status(e);
}

const char* strata_last_cuda_error(void) {
    return t_last_cuda == cudaSuccess ? "no error" : cudaGetErrorName(t_last_cuda);
}

const char* strata_status_str(strata_status s) {
    switch (s) {
        case STRATA_OK: return "STRATA_OK";
        case STRATA_EINVAL: return "STRATA_EINVAL: invalid argument";
        case STRATA_ECUDA: return "STRATA_ECUDA: CUDA launch or query failed";
        case STRATA_EUNSUPPORTED: return "STRATA_EUNSUPPORTED: not handled by this build";
        case STRATA_ETIMEOUT: return "STRATA_ETIMEOUT: a bounded device wait ran out";
        case STRATA_EBADROUTE: return "STRATA_EBADROUTE: expert id out of range";
        case STRATA_ERANGE: return "STRATA_ERANGE: a value left the fp16 operand range";
    }
    return "unknown strata_status";
}

}  // extern "C"

// ---------------------------------------------------------------------------
// A workspace that lives inside the library, for callers that cannot allocate
// device memory: a plugin whose host framework owns every device allocation
// and hands the plugin only its inputs and outputs, or an engine that must
// not call cudaMalloc (which may synchronise the device) on its serving path.
// It is one fixed 2 MiB array per device that loads the library, kept until
// the process exits, shared by every call of moe_layer_forward_static.

namespace {

constexpr size_t kStaticWsBytes = size_t(2) << 20;
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// The array's device address in the current device's context, looked up on
// every call (host code may not use the symbol itself as a device pointer).
// Nothing is cached, so a context torn down and made again (cudaDeviceReset)
// gets the address of its own copy of the array.
void* static_ws_address() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess) return nullptr;
    return p;
}

}  // namespace

extern "C" strata_status moe_layer_forward_static(const strata_moe_dims* dims,
                                                  const strata_moe_layer* layer,
                                                  const void* x_dev, int32_t T, int32_t* ids_dev,
                                                  float* weights_dev, float* shared_gate_dev,
                                                  void* out_dev, void* stream) {
    if (!dims_ok(dims) || T < 0 || !layer_ok(layer, kRouter | kRouted | kShared))
        return STRATA_EINVAL;
    if (T == 0) return STRATA_OK;
    if (!al16(x_dev) || !opt4(ids_dev) || !opt4(weights_dev) || !opt4(shared_gate_dev) ||
        !al16(out_dev))
        return STRATA_EINVAL;
    if (T > kDecodeMaxTokens || ws_layout(*dims, T).decode_end > kStaticWsBytes)
        return STRATA_EINVAL;
    void* ws = static_ws_address();
    if (ws == nullptr) return STRATA_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the error word must start at zero; every other region is written
    // before it is read
    if (cudaMemsetAsync(ws, 0, sizeof(Ctl), s) != cudaSuccess) return STRATA_ECUDA;
    return decode_layer(dims, layer, x_dev, T, nullptr, nullptr, ids_dev, weights_dev,
                        shared_gate_dev, out_dev, nullptr, ws, s);
}
