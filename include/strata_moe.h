/*
 * strata_moe.h -- C ABI of the GB300 (sm_103a) routed mixture-of-experts FFN
 * forward: router -> top-K -> int4-block-quantized SwiGLU experts -> weighted
 * combine with a sigmoid-gated shared expert.
 *
 * What the operation is (the pages describe it in engineering notes, never as
 * a formula; the plain reading taken here is stated with each call):
 *   Strata, "Qwen3.6-35B-A3B: pictures, several requests at once and speed",
 *   section "Speed": a 256-expert, top-8 MoE whose router and shared-expert
 *   gate are one product, SwiGLU experts, router top-k and grouping in one
 *   launch, the weighted sum of the experts ("the MoE end").  Section
 *   "Several requests at once": every routed expert two tokens share is read
 *   once for both.  PolyStrata, "Models and backends", section "What was
 *   tuned": a launch covers a call's experts together, one launch adds them up.
 *
 * Conventions for every call
 *   - Pointers named *_dev are device pointers; nothing else is.  The caller
 *     allocates every buffer; the library allocates nothing, frees nothing and
 *     never synchronises inside a forward call.  It keeps no pointer across
 *     calls.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) in call order.
 *   - `ws_dev` is a caller-owned device workspace of at least
 *     moe_workspace_bytes(dims, max_tokens) bytes, 256-byte aligned, created
 *     zero-filled once (the library keeps it consistent afterwards).  Two
 *     calls that may run at the same time (two streams) must not share a
 *     workspace: the pages report silent corruption from exactly that sharing
 *     (colibri, "qwen36: CUDA VRAM expert tier", section "Placement").
 *   - Host-side validation comes first: an unsupported shape, a NULL or
 *     misaligned pointer, T < 0, T > the workspace's max_tokens or a too-small
 *     workspace returns STRATA_EINVAL with nothing launched.  T == 0 returns
 *     STRATA_OK and launches nothing.  A failed launch returns STRATA_ECUDA.
 *   - Kernels never trap.  A forced expert id outside [0, E) is skipped and
 *     latches STRATA_EBADROUTE in the workspace's error word; a bounded wait
 *     that runs out latches STRATA_ETIMEOUT (over any code latched before
 *     it: the other waits of the call then give up early); on the tensor-core path
 *     (STRATA_PATH_TC), an activation or h whose fp16 operand copy is not
 *     finite (|value| beyond 65504, or a non-finite input) latches
 *     STRATA_ERANGE and is written saturated (+-65504, 0 for a NaN), so the
 *     products stay finite, and a non-finite output (an expert output past
 *     the fp16 range among the causes) latches it too; the call's outputs
 *     are then not to be used.
 *     moe_get_device_status reads and clears the word.
 *   - Results are deterministic: ids, permutations and every floating sum are
 *     computed in a fixed order, with no floating-point atomics.
 *
 * Supported shapes: group == 32; hidden H a multiple of 256 in [256, 4096];
 * n_experts E in [1, 1024]; top_k K in [1, min(E, 16)]; inter I and
 * shared_inter Is each one of 64, 128, 256, 512, 1024.
 *
 * Packed-weight layout (16-byte aligned planes; a layer is one caller-owned
 * allocation or several, any order):
 *   router      bf16 [E+1][H]: row e < E is expert e's router row, row E is
 *               the shared-expert gate vector (one more row of the same
 *               product, as on the Strata page).
 *   router_bias fp32 [E] added to the logits before selection, or NULL.
 *   gu_q        uint8 [E][2I][H/2]   gate/up rows interleaved: row 2i is
 *               gate row i, row 2i+1 is up row i.
 *   gu_s        fp16  [E][2I][H/32]  one scale per 32 consecutive inputs.
 *   dn_q        uint8 [E][H][I/2],  dn_s fp16 [E][H][I/32]
 *   sh_gu_q/s, sh_dn_q/s: the same for the one shared expert with Is.
 *   int4 nibbles: byte b of a row holds element 2b in bits 0..3 and element
 *   2b+1 in bits 4..7, offset-binary: weight = scale * (nibble - 8), the
 *   signed value "one XOR with 0x88888888" yields ("Every Public GGUF of This
 *   Model Is Missing Its Head", section 5).  Symmetric: no zero point.
 */
#ifndef STRATA_MOE_H
#define STRATA_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define STRATA_API __attribute__((visibility("default")))
#else
#define STRATA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    STRATA_OK = 0,
    STRATA_EINVAL = 1,        /* bad argument; nothing launched            */
    STRATA_ECUDA = 2,         /* a CUDA launch or query failed             */
    STRATA_EUNSUPPORTED = 3,  /* valid request this build does not handle  */
    STRATA_ETIMEOUT = 4,      /* a bounded device wait ran out (latched)   */
    STRATA_EBADROUTE = 5,     /* a forced expert id was out of range (latched) */
    STRATA_ERANGE = 6         /* a tensor-core fp16 operand overflowed (latched) */
} strata_status;

typedef struct {
    int32_t hidden;        /* H */
    int32_t n_experts;     /* E */
    int32_t top_k;         /* K */
    int32_t inter;         /* I, routed expert intermediate size */
    int32_t shared_inter;  /* Is, shared expert intermediate size */
    int32_t group;         /* scale group along the input axis; must be 32 */
} strata_moe_dims;

typedef struct {
    const void* router_dev;          /* bf16 [E+1][H] */
    const float* router_bias_dev;    /* fp32 [E] or NULL */
    const uint8_t* gu_q_dev;   const uint16_t* gu_s_dev;
    const uint8_t* dn_q_dev;   const uint16_t* dn_s_dev;
    const uint8_t* sh_gu_q_dev; const uint16_t* sh_gu_s_dev;
    const uint8_t* sh_dn_q_dev; const uint16_t* sh_dn_s_dev;
} strata_moe_layer;

/* Bytes of workspace the calls below need for up to max_tokens tokens of a
 * layer of shape *dims; 0 when the shape is unsupported or max_tokens < 1. */
STRATA_API size_t moe_workspace_bytes(const strata_moe_dims* dims, int32_t max_tokens);

/* The T at and below which the stage calls (moe_route ... moe_combine), the
 * moe_decode_* calls and moe_layer_forward_static take the decode (GEMV)
 * kernels; above it they take the tcgen05 grouped-GEMM (prefill) kernels. */
STRATA_API int32_t moe_decode_max_tokens(void);

/* The T at and below which the whole-layer calls (moe_layer_forward,
 * moe_layer_forward_routed, moe_block_forward, moe_stack_forward) take the
 * three decode kernels when the persistent kernel does not take the call
 * (see moe_layer_path); above it they take the tcgen05 kernels, unless the
 * shape does not allow those (hidden % 256 != 0 or an intermediate size
 * below 256), when the decode kernels serve up to moe_decode_max_tokens(). */
STRATA_API int32_t moe_layer_decode_max_tokens(void);

/* Input RMSNorm, unit weight:  x[t][h] = bf16( r[t][h] / sqrt(mean_h r^2 + eps) ).
 * Strata "Speed": "add+norm+q8_1 in one launch" is the norm in front of the
 * MoE; this build keeps bf16 activations.
 * r_dev fp32 [T][H] (in), x_dev bf16 [T][H] (out). */
STRATA_API strata_status moe_rmsnorm(const float* r_dev, int32_t T, int32_t H, float eps, void* x_dev,
                          void* stream);

/* Router product, top-K selection and renormalised softmax, shared gate.
 *   logits[t][e] = sum_h x[t][h] router[e][h] + bias[e]     (fp32 sums)
 *   ids[t][.]    the K largest logits, ties to the lower expert id (PolyStrata
 *                "What was tuned": the first of equal values wins), stored in
 *                ascending expert id
 *   weights[t][k] = exp(l_k - m) / sum_k' exp(l_k' - m) over the selected,
 *                m the largest selected logit (softmax over all E followed by
 *                renormalisation over the K selected is the same number)
 *   shared_gate[t] = 1 / (1 + exp(-sum_h x[t][h] router[E][h]))
 * x_dev bf16 [T][H]; ids_dev int32 [T][K]; weights_dev fp32 [T][K];
 * shared_gate_dev fp32 [T]; logits_dev fp32 [T][E] or NULL. */
STRATA_API strata_status moe_route(const strata_moe_dims* dims, const strata_moe_layer* layer,
                        const void* x_dev, int32_t T, int32_t* ids_dev, float* weights_dev,
                        float* shared_gate_dev, float* logits_dev, void* ws_dev,
                        size_t ws_bytes, void* stream);

/* Bucketing of the T*K (token, k) pairs by expert (Strata "Speed": router
 * top-k and grouping; the one-thread `k_group` the page found slow is a
 * block-parallel counting sort here):
 *   counts[e]      number of pairs routed to e
 *   offsets[0..E]  exclusive prefix sum of counts, offsets[E] = T*K
 *   perm[slot]     t*K + k, slots of one expert in ascending t (stable)
 *   inv_perm[t*K+k] = slot
 * ids_dev int32 [T][K] from any source (forced routing allowed); an id out of
 * range is skipped and latches STRATA_EBADROUTE. */
STRATA_API strata_status moe_permute(const strata_moe_dims* dims, const int32_t* ids_dev, int32_t T,
                          int32_t* counts_dev, int32_t* offsets_dev, int32_t* perm_dev,
                          int32_t* inv_perm_dev, void* ws_dev, size_t ws_bytes, void* stream);

/* Routed experts' gate/up product and SwiGLU (every expert's weights are read
 * once for all tokens routed to it: Strata "Several requests at once").
 * For each slot s of expert e (offsets) and token t = perm[s] / K:
 *   g_i = sum_h x[t][h] Wg[e][i][h],  u_i = sum_h x[t][h] Wu[e][i][h]
 *   h[s][i] = g_i / (1 + exp(-g_i)) * u_i
 * with W = fp16 scale * (nibble - 8).  h_dev fp32 [T*K][I] (out).
 * Above moe_decode_max_tokens() the product runs on the tensor cores with
 * fp16 operands (x rounded to fp16) and fp32 accumulation; at and below it,
 * on the CUDA cores in fp32.  The same holds for the down product and the
 * shared expert below (h rounded to fp16 there).  An expert whose offsets
 * leave [0, T*K] is skipped and latches STRATA_EBADROUTE. */
STRATA_API strata_status moe_expert_gate_up(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                 const void* x_dev, int32_t T, const int32_t* offsets_dev,
                                 const int32_t* perm_dev, float* h_dev, void* ws_dev,
                                 size_t ws_bytes, void* stream);

/* Routed experts' down product: y[s][o] = sum_i h[s][i] Wd[e][o][i] for every
 * slot s of expert e.  h_dev fp32 [T*K][I] (in), y_dev bf16 [T*K][H] (out). */
STRATA_API strata_status moe_expert_down(const strata_moe_dims* dims, const strata_moe_layer* layer,
                              const float* h_dev, int32_t T, const int32_t* offsets_dev,
                              void* y_dev, void* ws_dev, size_t ws_bytes, void* stream);

/* moe_expert_gate_up followed by moe_expert_down, h kept in the workspace.
 * y_dev bf16 [T*K][H], permuted (slot) order. */
STRATA_API strata_status moe_expert_ffn(const strata_moe_dims* dims, const strata_moe_layer* layer,
                             const void* x_dev, int32_t T, const int32_t* offsets_dev,
                             const int32_t* perm_dev, void* y_dev, void* ws_dev,
                             size_t ws_bytes, void* stream);

/* Shared expert and weighted combine ("the MoE end", Strata "Speed"; "one
 * launch adds up a call's experts", PolyStrata "What was tuned"):
 *   S[t]        the shared SwiGLU expert on x[t] (same arithmetic, Is)
 *   out[t][o] = bf16( sum_{k ascending} w[t][k] y[inv[t*K+k]][o]
 *                     + shared_gate[t] S[t][o] )       (fp32 sum)
 * y_dev bf16 [T*K][H]; inv_perm_dev int32 [T*K]; weights_dev fp32 [T][K];
 * shared_gate_dev fp32 [T]; out_dev bf16 [T][H]. */
STRATA_API strata_status moe_combine(const strata_moe_dims* dims, const strata_moe_layer* layer,
                          const void* x_dev, int32_t T, const void* y_dev,
                          const int32_t* inv_perm_dev, const float* weights_dev,
                          const float* shared_gate_dev, void* out_dev, void* ws_dev,
                          size_t ws_bytes, void* stream);

/* The whole layer: route, permute, experts, shared expert, combine.  Which
 * kernels run is moe_layer_path(dims, T): for one token ONE persistent
 * kernel (one CTA per SM; the router product, top-K and bucketing, the
 * routed gate/up, the down products and the combine, values passing between
 * CTAs as tagged words in the workspace; PolyStrata, "Models and backends",
 * section "What was tuned": decode was launch-bound at ~35 launches a
 * layer), else three decode kernels or the tcgen05 prefill kernels.
 * ids_dev / weights_dev / shared_gate_dev receive the routing when non-NULL.
 * out_dev bf16 [T][H]. */
STRATA_API strata_status moe_layer_forward(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                const void* x_dev, int32_t T, int32_t* ids_dev,
                                float* weights_dev, float* shared_gate_dev, void* out_dev,
                                void* ws_dev, size_t ws_bytes, void* stream);

/* As moe_layer_forward, but with the routing forced: ids_dev / weights_dev
 * (in) replace the router's choice; shared_gate is still computed. */
STRATA_API strata_status moe_layer_forward_routed(const strata_moe_dims* dims,
                                       const strata_moe_layer* layer, const void* x_dev,
                                       int32_t T, const int32_t* ids_dev,
                                       const float* weights_dev, void* out_dev, void* ws_dev,
                                       size_t ws_bytes, void* stream);

/* As moe_layer_forward, with tail-skip (PolyStrata, "Models and backends",
 * section "What was tuned"): in a decode window (T <= moe_decode_max_tokens())
 * an expert that every token of the call ranks at place tail_skip + 1 or
 * later of its top_k picks is not computed; the picks that stay keep the
 * router's weights (no renormalisation).  A pick's place counts its token's
 * picks with a larger weight, or an equal weight and a lower id.  The
 * window runs on the decode kernels whatever T is.  A prompt batch
 * (T > moe_decode_max_tokens()) is not touched and runs as
 * moe_layer_forward.  tail_skip = 0 or >= top_k leaves every pick.
 *   forced_ids_dev / forced_weights_dev: both NULL to route, or both given
 *     to force the routing (the places are then those of the given weights).
 *   ids_dev / weights_dev / shared_gate_dev (out, optional): the routing;
 *     the weights of left-out picks are written as 0, their ids as chosen.
 * Changes the layer's result by design: not a drop-in for the exact call.
 * STRATA_EINVAL for tail_skip < 0 or one of the forced pointers alone. */
STRATA_API strata_status moe_layer_forward_tail_skip(const strata_moe_dims* dims,
                                          const strata_moe_layer* layer, const void* x_dev,
                                          int32_t T, int32_t tail_skip,
                                          const int32_t* forced_ids_dev,
                                          const float* forced_weights_dev, int32_t* ids_dev,
                                          float* weights_dev, float* shared_gate_dev,
                                          void* out_dev, void* ws_dev, size_t ws_bytes,
                                          void* stream);

/* One residual MoE block of a layer stack:
 *   x = bf16(rmsnorm(resid, eps));  out = layer(x);  resid += float(out)
 * On the persistent kernel (moe_layer_path) the norm runs inside it. 
 * resid_dev fp32 [T][H] (in/out).  ids_dev / weights_dev: NULL to route, or
 * both non-NULL to force the routing.  x_out_dev / out_dev: optional bf16
 * [T][H] copies of the block's input and output (NULL: workspace only). */
STRATA_API strata_status moe_block_forward(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                float* resid_dev, int32_t T, float eps, const int32_t* ids_dev,
                                const float* weights_dev, void* x_out_dev, void* out_dev,
                                void* ws_dev, size_t ws_bytes, void* stream);

/* A stack of n_layers residual MoE blocks, layer after layer:
 *   for l in 0..n_layers-1:  x = bf16(rmsnorm(resid, eps));  resid += float(layer_l(x))
 * layers: HOST array of n_layers layer descriptors (device pointers inside);
 * read during the call only.  resid_dev fp32 [T][H] (in/out); ids_dev /
 * weights_dev: NULL to route every layer, or both int32 / fp32
 * [n_layers][T][K] to force the routing; out_dev: NULL or bf16 [T][H], the
 * last layer's output ("qwen36: CUDA VRAM expert tier", section
 * "Placement": a token's routed experts are 40 layers of top-8).  Where
 * moe_layer_path(dims, T) is STRATA_PATH_PERSISTENT the whole stack runs as
 * one persistent kernel per 40 layers: each layer's RMSNorm, routing,
 * experts and residual add inside it, and each CTA's share of the next
 * layer's router and shared-expert rows requested while the current layer
 * streams its experts.  Otherwise one moe_block_forward per layer. */
STRATA_API strata_status moe_stack_forward(const strata_moe_dims* dims,
                                           const strata_moe_layer* layers, int32_t n_layers,
                                           float* resid_dev, int32_t T, float eps,
                                           const int32_t* ids_dev, const float* weights_dev,
                                           void* out_dev, void* ws_dev, size_t ws_bytes,
                                           void* stream);

/* The three kernels of the decode path (T <= moe_decode_max_tokens()), as
 * separate calls; moe_layer_forward is the three in a row.  They pass their
 * state through the workspace (logits, the shared expert's SwiGLU vectors,
 * the routing, the bucketing and a plan of the touched experts, the routed
 * SwiGLU vectors), so they take the same workspace and T, in this order.
 *   moe_decode_route        the router product (all E+1 rows, or with
 *                           forced != 0 only the shared-gate row) and the
 *                           shared expert's gate/up + SwiGLU, one kernel.
 *   moe_decode_gate_up      top-K, softmax and sigmoid gate of every token
 *                           (or the forced ids/weights: both NULL or both
 *                           given), the bucketing, then every touched
 *                           expert's gate/up + SwiGLU, one kernel.
 *                           ids_dev / weights_dev / shared_gate_dev: optional
 *                           copies of the routing.
 *   moe_decode_down_combine every touched expert's down product, the shared
 *                           expert's, and the weighted combine into out_dev
 *                           (bf16 [T][H]); resid_dev (fp32 [T][H], optional)
 *                           gets += the bf16 output. */
STRATA_API strata_status moe_decode_route(const strata_moe_dims* dims, const strata_moe_layer* layer,
                                          const void* x_dev, int32_t T, int32_t forced,
                                          void* ws_dev, size_t ws_bytes, void* stream);
STRATA_API strata_status moe_decode_gate_up(const strata_moe_dims* dims,
                                            const strata_moe_layer* layer, const void* x_dev,
                                            int32_t T, const int32_t* forced_ids_dev,
                                            const float* forced_weights_dev, int32_t* ids_dev,
                                            float* weights_dev, float* shared_gate_dev,
                                            void* ws_dev, size_t ws_bytes, void* stream);
STRATA_API strata_status moe_decode_down_combine(const strata_moe_dims* dims,
                                                 const strata_moe_layer* layer, int32_t T,
                                                 void* out_dev, float* resid_dev, void* ws_dev,
                                                 size_t ws_bytes, void* stream);

/* moe_layer_forward without a caller-supplied workspace.  The pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory -- a plugin whose host framework owns every device allocation and
 * hands it only inputs and outputs, or a serving path that must not call
 * cudaMalloc.  The workspace is a fixed 2 MiB array inside the library: every
 * GPU that loads the library holds it until the process exits, and every call
 * of this function on a device uses the same array.
 *   - Runs the decode kernels at every T it takes.  Limits: T <=
 *     moe_decode_max_tokens() and the decode kernels' part of the workspace
 *     <= 2 MiB (every decode T of the 2048-hidden, 256-expert, top-8 shape
 *     fits); a larger request returns STRATA_EINVAL with nothing launched.
 *   - Every call looks up the array's device address in the current
 *     device's context (cudaGetSymbolAddress; nothing cached, so a context
 *     made again after cudaDeviceReset gets its own copy).  The first call on
 *     a device loads the library's kernels there: make it before any stream
 *     capture.  No call allocates or frees anything.
 *   - Calls that may overlap on the GPU (several streams, or several host
 *     threads on one device) race on the shared array and give wrong results:
 *     serialise them, or use moe_layer_forward with one workspace each.
 *   - Device-side checks latch into the array's own error word, which each
 *     call clears first and this call cannot report; use moe_layer_forward and
 *     moe_get_device_status where those checks matter.
 * Arguments as moe_layer_forward. */
STRATA_API strata_status moe_layer_forward_static(const strata_moe_dims* dims,
                                                  const strata_moe_layer* layer,
                                                  const void* x_dev, int32_t T,
                                                  int32_t* ids_dev, float* weights_dev,
                                                  float* shared_gate_dev, void* out_dev,
                                                  void* stream);

/* Measurement: runs moe_layer_forward once with a CUDA event recorded after
 * every kernel launch, synchronises `stream`, and writes each kernel's
 * duration in microseconds to us[0..max_n) in launch order; *n_out gets the
 * number of kernels.  The events serialise the kernels, so each duration is
 * the kernel alone.  Order, by moe_layer_path: the persistent kernel (one);
 * the decode kernels (three): route, gate/up, down+combine; tcgen05 kernels (nine):
 * router GEMM, top-K, count, scan, scatter, gather, gate/up GEMM, down GEMM,
 * combine -- seven at T <= 32, where count, scan and scatter are one
 * bucketing kernel. */
STRATA_API strata_status moe_layer_profile(const strata_moe_dims* dims,
                                           const strata_moe_layer* layer, const void* x_dev,
                                           int32_t T, void* out_dev, void* ws_dev,
                                           size_t ws_bytes, void* stream, float* us,
                                           int32_t max_n, int32_t* n_out);

/* Which kernels a whole-layer call (moe_layer_forward, _routed,
 * moe_block_forward, moe_stack_forward) runs for T tokens of this shape on
 * the current device: STRATA_PATH_PERSISTENT (one persistent kernel a call;
 * a stack, one per 40 layers), STRATA_PATH_DECODE (three decode kernels a
 * layer, plus the RMSNorm kernel in a block), STRATA_PATH_TC (the tcgen05
 * prefill kernels), or 0 for an unsupported shape or T < 1.  forced != 0
 * asks for a call with forced routing.  Host only; no GPU work. */
#define STRATA_PATH_PERSISTENT 1
#define STRATA_PATH_DECODE 2
#define STRATA_PATH_TC 3
STRATA_API int32_t moe_layer_path(const strata_moe_dims* dims, int32_t T, int32_t forced);

/* The bucketing of the last whole-layer call (moe_layer_forward or _routed,
 * any path) made on this workspace with this T: copies counts int32 [E],
 * offsets int32 [E+1], perm int32 [T*K] and inv_perm int32 [T*K] (layout as
 * moe_permute) out of the workspace, on `stream`.  For tests and debugging:
 * it shows the bucketing the layer's own kernels built, which the stage call
 * moe_permute does not run.  STRATA_EINVAL for a bad argument. */
STRATA_API strata_status moe_layer_bucketing(const strata_moe_dims* dims, int32_t T,
                                             const void* ws_dev, size_t ws_bytes,
                                             int32_t* counts_dev, int32_t* offsets_dev,
                                             int32_t* perm_dev, int32_t* inv_perm_dev,
                                             void* stream);

/* Synchronises `stream`, returns the status latched in the workspace's error
 * word (STRATA_OK when none) and clears the word.  For tests and debugging;
 * it is the one call that synchronises. */
STRATA_API strata_status moe_get_device_status(void* ws_dev, void* stream);

/* Testing hook: the number of polls after which a grid-wide barrier of the
 * persistent kernel gives up, latches STRATA_ETIMEOUT in the workspace's
 * error word and lets the kernel run on to its end (with wrong values, but
 * without hanging).  0 restores the default (~2^21 polls, a second or two).
 * Applies to launches made after the call, from any host thread.  Copies
 * into shared memory are always waited for in full. */
STRATA_API void strata_set_grid_wait_limit(uint32_t polls);

/* Phase timestamps of the persistent kernel (the one-token layer and the
 * stack, moe_layer_path() == 1), for a library built with phase tracing
 * (quantized_moe_expert_fwd_gb300.build.build(trace=True), which compiles
 * with STRATA_PX_TRACE; the default library records none and returns
 * STRATA_EUNSUPPORTED).  Copies min(bytes, 512 KiB) of the last launch's
 * record to host memory `host`: uint64 global-timer readings in ns, laid out
 * [CTA 0..1023][slot 0..3][point 0..15]; slots are the launch's layers 0, 1,
 * n/2 and n-1 (the first match), points:
 *   0 CTA initialised (slot 0 only)      1 grid dependency resolved (slot 0)
 *   2 token row in shared memory         3 router rows and shared pairs done
 *   4 token 0's logits all seen          5 token 0's top-K and gate done
 *   6 plan published                     7 the CTA's gate/up stages done
 *   8 SwiGLU rows staged                 9 down products done
 *  10 combined                          11 producer: plan seen
 *  12 producer: gate/up copies issued   13 producer: down copies issued
 * (unused entries are left as they were).  Synchronises the device.
 * Returns STRATA_EINVAL for a NULL `host` or zero `bytes`, STRATA_ECUDA when
 * the copy fails. */
STRATA_API strata_status strata_px_trace_read(void* host, size_t bytes);

/* Static, human-readable name of a status. */
STRATA_API const char* strata_status_str(strata_status s);

/* Name of the last CUDA error behind a STRATA_ECUDA returned to the calling
 * host thread ("no error" when there was none); static storage. */
STRATA_API const char* strata_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* STRATA_MOE_H */
