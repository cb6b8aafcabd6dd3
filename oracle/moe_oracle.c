/*
 * moe_oracle.c -- plain, slow, fp32 CPU reference of the routed MoE FFN
 * forward (router -> top-K -> int4-block-quantized SwiGLU experts -> weighted
 * combine + sigmoid-gated shared expert).
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the bench's CPU
 * baseline leg call this file.  It shares no code, header, table or helper
 * with the CUDA library, and it never reads anything the CUDA library wrote.
 *
 * Arithmetic rules, chosen so that a reader can check every line by eye:
 *   - every float is fp32; every dot product is one serial sum in ascending
 *     index order; no blocking, no reassociation, no fused multiply-add
 *     (the build passes -ffp-contract=off so x86 and Arm give the same bits);
 *   - int4 weights are dequantised exactly: fp16 scale * (nibble - 8) is exact
 *     in fp32;
 *   - bf16 and fp16 are decoded from their IEEE bit layouts here.
 *
 * Sources.  The pages this follows are engineering notes, not a specification:
 *   - Strata, "Qwen3.6-35B-A3B: pictures, several requests at once and speed",
 *     section "Speed": the router and the shared-expert gate are one product
 *     (one more router row), the experts are SwiGLU, routing is top-k with
 *     grouping of the selected experts.
 *   - PolyStrata, "Models and backends", section "What was tuned": among equal
 *     scores the first (lowest index) one wins; ties here go to the lower
 *     expert id.
 *   - "Every Public GGUF of This Model Is Missing Its Head", section 5: raw Q4
 *     nibbles are offset-binary (XOR with 8 gives the signed value), the
 *     convention of the packed layout.
 * Where the pages print no formula (the softmax, its renormalisation, the
 * sigmoid gate, the scale-group axis) the plainest reading is taken:
 *   w_k = exp(l_k - m) / sum_k' exp(l_k' - m) over the K selected logits,
 *   sigma = 1 / (1 + exp(-s)) multiplying the whole shared-expert output,
 *   one fp16 scale per 32 consecutive input (reduction) elements of a row.
 *
 * Parity of this file against the pages is unpinned: they print no value of
 * this computation.  Its pins are brute force, closed forms, invariants and
 * hand-computed packed bytes (tests/test_oracle_*.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* ---------------------------------------------------------------- formats */

/* bf16: the upper 16 bits of an IEEE binary32. */
ORC_API float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even; NaN stays NaN. */
ORC_API uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
ORC_API float orc_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);                 /* zero and subnormals */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

ORC_API void orc_round_bf16(int64_t n, const float* in, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------- dequantise */

/* Signed value of element j of a packed int4 row: byte j/2 holds element 2b
 * in bits 0..3 and element 2b+1 in bits 4..7, offset-binary (u - 8). */
ORC_API int orc_nibble(const uint8_t* q, int j) {
    uint8_t byte = q[j >> 1];
    int u = (j & 1) ? (byte >> 4) : (byte & 0x0f);
    return u - 8;
}

/* out[j] = scale[j/32] * q_j for j < n (exact in fp32). */
ORC_API void orc_dequant_row(const uint8_t* q, const uint16_t* s, int n, float* out) {
    for (int j = 0; j < n; ++j)
        out[j] = orc_f16_to_f32(s[j / 32]) * (float)orc_nibble(q, j);
}

/* rows x cols matrix from its packed planes (row stride cols/2 bytes and
 * cols/32 scales). */
ORC_API void orc_dequant_matrix(const uint8_t* q, const uint16_t* s, int rows, int cols,
                                float* out) {
    for (int r = 0; r < rows; ++r)
        orc_dequant_row(q + (size_t)r * (cols / 2), s + (size_t)r * (cols / 32), cols,
                        out + (size_t)r * cols);
}

/* ---------------------------------------------------------------- RMSNorm */

/* x[t] = bf16( r[t] / sqrt(mean(r[t]^2) + eps) ), unit weight. */
ORC_API void orc_rmsnorm(int T, int H, const float* r, float eps, uint16_t* x) {
    for (int t = 0; t < T; ++t) {
        const float* rt = r + (size_t)t * H;
        float ss = 0.0f;
        for (int h = 0; h < H; ++h) ss += rt[h] * rt[h];
        float denom = sqrtf(ss / (float)H + eps);
        for (int h = 0; h < H; ++h) x[(size_t)t * H + h] = orc_f32_to_bf16(rt[h] / denom);
    }
}

/* ----------------------------------------------------------------- router */

/* logits[t][e] = sum_h x[t][h] * router[e][h] (+ bias[e]) for e < E;
 * gate_logit[t] = sum_h x[t][h] * router[E][h]  (the shared gate row). */
ORC_API void orc_router(int T, int H, int E, const uint16_t* x, const uint16_t* router,
                        const float* bias, float* logits, float* gate_logit) {
    for (int t = 0; t < T; ++t) {
        const uint16_t* xt = x + (size_t)t * H;
        for (int e = 0; e <= E; ++e) {
            const uint16_t* we = router + (size_t)e * H;
            float acc = 0.0f;
            for (int h = 0; h < H; ++h) acc += orc_bf16_to_f32(xt[h]) * orc_bf16_to_f32(we[h]);
            if (e < E)
                logits[(size_t)t * E + e] = acc + (bias ? bias[e] : 0.0f);
            else
                gate_logit[t] = acc;
        }
    }
}

/* "a beats b": larger logit, or equal logit and lower index. */
static int orc_beats(float la, int a, float lb, int b) {
    return la > lb || (la == lb && a < b);
}

/* Top-K selection and renormalised softmax for each token.
 *   ids[t][.]  the K winners in ascending expert id
 *   w[t][k]    exp(l_k - m) / sum exp(l_k' - m), m = largest selected logit,
 *              sum taken in ascending expert id
 *   gap[t]     l_(K) - l_(K+1) on the sorted logits (+inf when E == K):
 *              how far the selection is from a tie */
ORC_API void orc_select(int T, int E, int K, const float* logits, int32_t* ids, float* w,
                        float* gap) {
    int* order = (int*)malloc(sizeof(int) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        /* selection sort of the first K+1 places by (logit desc, id asc) */
        for (int e = 0; e < E; ++e) order[e] = e;
        int places = (K + 1 < E) ? K + 1 : E;
        for (int p = 0; p < places; ++p) {
            int best = p;
            for (int q = p + 1; q < E; ++q)
                if (orc_beats(l[order[q]], order[q], l[order[best]], order[best])) best = q;
            int tmp = order[p]; order[p] = order[best]; order[best] = tmp;
        }
        if (gap) gap[t] = (K < E) ? l[order[K - 1]] - l[order[K]] : INFINITY;
        /* the K winners in ascending id */
        int32_t* it = ids + (size_t)t * K;
        for (int k = 0; k < K; ++k) it[k] = order[k];
        for (int a = 1; a < K; ++a)
            for (int b = a; b > 0 && it[b - 1] > it[b]; --b) {
                int32_t tmp = it[b]; it[b] = it[b - 1]; it[b - 1] = tmp;
            }
        float m = l[order[0]];
        float sum = 0.0f;
        for (int k = 0; k < K; ++k) sum += expf(l[it[k]] - m);
        for (int k = 0; k < K; ++k) w[(size_t)t * K + k] = expf(l[it[k]] - m) / sum;
    }
    free(order);
}

ORC_API float orc_sigmoid(float s) { return 1.0f / (1.0f + expf(-s)); }

/* silu(g) * u, silu(g) = g / (1 + exp(-g)) */
ORC_API float orc_swiglu(float g, float u) { return g / (1.0f + expf(-g)) * u; }

/* ------------------------------------------------------------- permutation */

/* Bucket the T*K (token, slot) pairs by expert: counts[e], offsets[0..E]
 * (exclusive scan, offsets[E] = T*K), perm[slot] = t*K + k with slots of one
 * expert in ascending t, inv[t*K + k] = slot.  A stable counting sort. */
ORC_API void orc_permute(int T, int K, int E, const int32_t* ids, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int p = 0; p < T * K; ++p) counts[ids[p]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int p = 0; p < T * K; ++p) {
        int e = ids[p];
        int slot = offsets[e] + fill[e]++;
        perm[slot] = p;
        inv[p] = slot;
    }
    free(fill);
}

/* -------------------------------------------------------------- expert FFN */

/* y = W x for a dense row-major W [rows][cols], each row one serial sum in
 * ascending column order.  Four rows are evaluated side by side only so the
 * CPU overlaps their independent sums; each row's own order is unchanged. */
static void orc_matvec(int rows, int cols, const float* W, const float* x, float* y) {
    int r = 0;
    for (; r + 4 <= rows; r += 4) {
        const float* w0 = W + (size_t)(r + 0) * cols;
        const float* w1 = W + (size_t)(r + 1) * cols;
        const float* w2 = W + (size_t)(r + 2) * cols;
        const float* w3 = W + (size_t)(r + 3) * cols;
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        for (int c = 0; c < cols; ++c) {
            a0 += w0[c] * x[c];
            a1 += w1[c] * x[c];
            a2 += w2[c] * x[c];
            a3 += w3[c] * x[c];
        }
        y[r] = a0; y[r + 1] = a1; y[r + 2] = a2; y[r + 3] = a3;
    }
    for (; r < rows; ++r) {
        const float* wr = W + (size_t)r * cols;
        float a = 0.0f;
        for (int c = 0; c < cols; ++c) a += wr[c] * x[c];
        y[r] = a;
    }
}

/* One SwiGLU expert on one token, weights already dequantised:
 *   Wgu [2I][H], row 2i = gate row i, row 2i+1 = up row i;  Wd [H][I].
 *   g = Wgu[2i] . x, u = Wgu[2i+1] . x, h_i = silu(g) u, y = Wd h.
 * gu is scratch of 2I floats. */
ORC_API void orc_expert_dense(int H, int I, const float* x, const float* Wgu, const float* Wd,
                              float* gu, float* h, float* y) {
    orc_matvec(2 * I, H, Wgu, x, gu);
    for (int i = 0; i < I; ++i) h[i] = orc_swiglu(gu[2 * i], gu[2 * i + 1]);
    orc_matvec(H, I, Wd, h, y);
}

typedef struct {
    const uint16_t* router;       /* bf16 [E+1][H] */
    const float* router_bias;     /* [E] or NULL */
    const uint8_t* gu_q;  const uint16_t* gu_s;       /* [E][2I][H/2], [E][2I][H/32] */
    const uint8_t* dn_q;  const uint16_t* dn_s;       /* [E][H][I/2],  [E][H][I/32]  */
    const uint8_t* sh_gu_q; const uint16_t* sh_gu_s;  /* [2Is][H/2], [2Is][H/32] */
    const uint8_t* sh_dn_q; const uint16_t* sh_dn_s;  /* [H][Is/2],  [H][Is/32]  */
} orc_layer;

/* The whole layer for T tokens.
 *   x      bf16 [T][H] (the normalised input)
 *   force  0: route here (ids, w, gap written);  1: use the given ids and w
 *   ids    [T][K] ascending per token; w [T][K]
 *   sig    [T] out: sigmoid(shared gate logit)
 *   out    [T][H] out, fp32:
 *            out[t][o] = sum_{k asc} w[t][k] y_k[o] + sig[t] S[t][o]
 *   y      optional [T][K][H] out: each selected expert's output
 *   h      optional [T][K][I] out: each selected expert's SwiGLU vector
 *   sh_y   optional [T][H] out: the shared expert's output S
 *   logits optional [T][E] out (only when force == 0)
 * Returns 0, or 1 when a forced id is out of range. */
ORC_API int orc_moe_forward(int H, int E, int K, int I, int Is, const orc_layer* L, int T,
                            const uint16_t* x, int force, int32_t* ids, float* w, float* gap,
                            float* sig, float* out, float* y, float* h, float* sh_y,
                            float* logits, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    float* lg = (float*)malloc(sizeof(float) * (size_t)T * E);
    float* gl = (float*)malloc(sizeof(float) * (size_t)T);
    orc_router(T, H, E, x, L->router, L->router_bias, lg, gl);
    if (!force) orc_select(T, E, K, lg, ids, w, gap);
    if (logits && !force) memcpy(logits, lg, sizeof(float) * (size_t)T * E);
    for (int p = 0; p < T * K; ++p)
        if (ids[p] < 0 || ids[p] >= E) { free(lg); free(gl); return 1; }
    for (int t = 0; t < T; ++t) sig[t] = orc_sigmoid(gl[t]);

    float* xf = (float*)malloc(sizeof(float) * (size_t)T * H);
    for (size_t i = 0; i < (size_t)T * H; ++i) xf[i] = orc_bf16_to_f32(x[i]);
    float* ybuf = y ? y : (float*)malloc(sizeof(float) * (size_t)T * K * H);
    float* sbuf = sh_y ? sh_y : (float*)malloc(sizeof(float) * (size_t)T * H);

    /* routed experts: each expert dequantised once, then every (t, k) that
     * selected it, in ascending t */
    #pragma omp parallel
    {
        float* Wgu = (float*)malloc(sizeof(float) * (size_t)2 * I * H);
        float* Wd = (float*)malloc(sizeof(float) * (size_t)H * I);
        float* gu = (float*)malloc(sizeof(float) * (size_t)2 * I);
        float* hv = (float*)malloc(sizeof(float) * (size_t)I);
        #pragma omp for schedule(dynamic, 1)
        for (int e = 0; e < E; ++e) {
            int loaded = 0;
            for (int p = 0; p < T * K; ++p) {
                if (ids[p] != e) continue;
                if (!loaded) {
                    orc_dequant_matrix(L->gu_q + (size_t)e * 2 * I * (H / 2),
                                       L->gu_s + (size_t)e * 2 * I * (H / 32), 2 * I, H, Wgu);
                    orc_dequant_matrix(L->dn_q + (size_t)e * H * (I / 2),
                                       L->dn_s + (size_t)e * H * (I / 32), H, I, Wd);
                    loaded = 1;
                }
                int t = p / K;
                orc_expert_dense(H, I, xf + (size_t)t * H, Wgu, Wd, gu, hv,
                                 ybuf + (size_t)p * H);
                if (h) memcpy(h + (size_t)p * I, hv, sizeof(float) * (size_t)I);
            }
        }
        free(Wgu); free(Wd); free(gu); free(hv);
    }
    /* shared expert on every token */
    {
        float* Wgu = (float*)malloc(sizeof(float) * (size_t)2 * Is * H);
        float* Wd = (float*)malloc(sizeof(float) * (size_t)H * Is);
        orc_dequant_matrix(L->sh_gu_q, L->sh_gu_s, 2 * Is, H, Wgu);
        orc_dequant_matrix(L->sh_dn_q, L->sh_dn_s, H, Is, Wd);
        #pragma omp parallel
        {
            float* gu = (float*)malloc(sizeof(float) * (size_t)2 * Is);
            float* hv = (float*)malloc(sizeof(float) * (size_t)Is);
            #pragma omp for schedule(static)
            for (int t = 0; t < T; ++t)
                orc_expert_dense(H, Is, xf + (size_t)t * H, Wgu, Wd, gu, hv,
                                 sbuf + (size_t)t * H);
            free(gu); free(hv);
        }
        free(Wgu); free(Wd);
    }
    /* combine */
    for (int t = 0; t < T; ++t)
        for (int o = 0; o < H; ++o) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k)
                acc += w[(size_t)t * K + k] * ybuf[((size_t)t * K + k) * H + o];
            out[(size_t)t * H + o] = acc + sig[t] * sbuf[(size_t)t * H + o];
        }

    if (!y) free(ybuf);
    if (!sh_y) free(sbuf);
    free(xf); free(lg); free(gl);
    return 0;
}
