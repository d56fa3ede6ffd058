/*
 * moe_oracle.c -- CPU oracle for one quantized MoE decode step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this code. The product path (the CUDA library) does
 * not link, include or call it, and shares no header, helper or table with it.
 *
 * What it computes: for a cohort of n tokens, the router GEMV, softmax over
 * all experts, top-k, renormalisation of the k selected probabilities,
 * grouping of the (token, k) slots by expert, each selected expert's SwiGLU
 * MLP on affine 4-bit weights, and the weighted sum of each token's k expert
 * outputs.
 *
 * Sources (mlxcel GitHub issues):
 *   #1616 "perf(moe): batched decode scales 1.55x against 3.25x on dense"
 *     - Current Behavior: the decode MoE block is SwitchGLU (gate/up/down
 *       expert projections) followed by moe_weighted_sum over the k slots;
 *       qwen3-30b-a3b-4bit experts are "4-bit group 64".
 *     - Leading hypothesis: the slot grouping is a sort by expert id.
 *     - Implementation Notes: the parity reference is an all-f32 dense
 *       reference, with f32 partials and a single final rounding.
 *   #1859 "perf(moe): attribute the MoE decode gap at the M = 1 expert
 *     gather" - Problem/Background: the decode step gathers one expert row per
 *     (token, k) slot, which is what grouping removes.
 * The pages give no formula for the router, the 4-bit format or SwiGLU; the
 * readings taken here (softmax over all experts, then top-k, then
 * renormalise; MLX affine w = s*q + b with codes 0..15, low nibble first,
 * groups of 64 along the input dimension, bf16 s and b; silu(z) =
 * z / (1 + exp(-z))) are the plainest ones and are listed with the design
 * notes of this repository.
 *
 * Precision: all arithmetic in f32 (the pages' "all-f32" reference), sums in
 * ascending index order, one rounding to bf16 at the very end if asked.
 * Ties in top-k go to the lower expert index.
 *
 * Pins (what this code is checked against, all on the CPU): the quantiser's
 * round-trip bound on the original weights, a float64 brute-force dense
 * formulation built from library routines (numpy matmul, scipy softmax),
 * the E=1 and k=1 and k=E special cases, x=0, routing-weight sums, expert
 * storage-order and token-order permutations, identical tokens, a stable
 * sort for the grouping, and, for the final rounding, PyTorch's float32 to
 * bfloat16 cast plus round-to-nearest-even taken from its definition on
 * exact rational distances (ties, carries, subnormals, overflow, NaN).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_GROUP 64

static float bf16_widen(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t bf16_round_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))  /* NaN */
        return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

int oracle_set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Weight of input column j of one quantised row: w = s*q + b, where q is
 * nibble (j mod 8) of word j/8 and (s, b) is the bf16 pair of group j/64. */
static float dequant_at(const uint32_t *qrow, const uint16_t *srow,
                        const uint16_t *brow, int j) {
    uint32_t word = qrow[j / 8];
    float q = (float)((word >> (4 * (j % 8))) & 0xFu);
    float s = bf16_widen(srow[j / ORACLE_GROUP]);
    float b = bf16_widen(brow[j / ORACLE_GROUP]);
    return fmaf(s, q, b);
}

/* Weight of input column j of one 6-bit row. The row's codes form one
 * little-endian bit stream of bytes: code j occupies bits 6j .. 6j+5 (four codes
 * in three bytes); w = s*q + b with q in 0..63 and the bf16 pair of group j/64. */
static float dequant6_at(const uint8_t *qrow, const uint16_t *srow, const uint16_t *brow, int j) {
    int bit = 6 * j, byte = bit >> 3, sh = bit & 7;
    uint32_t v = qrow[byte];
    if (sh > 2) v |= (uint32_t)qrow[byte + 1] << 8;  /* the code spans two bytes */
    float q = (float)((v >> sh) & 0x3Fu);
    float s = bf16_widen(srow[j / ORACLE_GROUP]);
    float b = bf16_widen(brow[j / ORACLE_GROUP]);
    return fmaf(s, q, b);
}

/* Dequantise a [rows, cols] 6-bit plane (rows of 3*cols/4 bytes) to f32. */
void oracle_dequant6(const uint8_t *q, const uint16_t *s, const uint16_t *b,
                     int rows, int cols, float *out) {
    for (int r = 0; r < rows; ++r) {
        const uint8_t *qr = q + (size_t)r * (3 * cols / 4);
        const uint16_t *sr = s + (size_t)r * (cols / ORACLE_GROUP);
        const uint16_t *br = b + (size_t)r * (cols / ORACLE_GROUP);
        for (int j = 0; j < cols; ++j) out[(size_t)r * cols + j] = dequant6_at(qr, sr, br, j);
    }
}

/* Dequantise a [rows, cols] plane to f32. */
void oracle_dequant(const uint32_t *q, const uint16_t *s, const uint16_t *b,
                    int rows, int cols, float *out) {
    for (int r = 0; r < rows; ++r) {
        const uint32_t *qr = q + (size_t)r * (cols / 8);
        const uint16_t *sr = s + (size_t)r * (cols / ORACLE_GROUP);
        const uint16_t *br = b + (size_t)r * (cols / ORACLE_GROUP);
        for (int j = 0; j < cols; ++j) out[(size_t)r * cols + j] = dequant_at(qr, sr, br, j);
    }
}

/* Router: logits, softmax over all E experts, top-k (descending logit, ties to
 * the lower index), renormalise the k selected probabilities.
 * x [n,D], wr [E,D], bias [E] or NULL -> topk_idx [n,k], topk_w [n,k];
 * logits [n,E] and probs [n,E] are written when non-NULL. */
void oracle_route(int n, int E, int D, int k, const float *x, const float *wr,
                  const float *bias, int32_t *topk_idx, float *topk_w,
                  float *logits_out, float *probs_out) {
    float *l = (float *)malloc(sizeof(float) * (size_t)E);
    float *p = (float *)malloc(sizeof(float) * (size_t)E);
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    for (int t = 0; t < n; ++t) {
        const float *xt = x + (size_t)t * D;
        for (int e = 0; e < E; ++e) {
            const float *we = wr + (size_t)e * D;
            float acc = 0.0f;
            for (int d = 0; d < D; ++d) acc = fmaf(xt[d], we[d], acc);
            if (bias) acc += bias[e];
            l[e] = acc;
        }
        float m = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
        float z = 0.0f;
        for (int e = 0; e < E; ++e) { p[e] = expf(l[e] - m); z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] = p[e] / z;
        if (logits_out) memcpy(logits_out + (size_t)t * E, l, sizeof(float) * (size_t)E);
        if (probs_out) memcpy(probs_out + (size_t)t * E, p, sizeof(float) * (size_t)E);

        memset(taken, 0, (size_t)E);
        float psum = 0.0f;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;  /* strict: ties keep lower e */
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
            psum += p[best];
        }
        for (int j = 0; j < k; ++j)
            topk_w[(size_t)t * k + j] = p[topk_idx[(size_t)t * k + j]] / psum;
    }
    free(l); free(p); free(taken);
}

/* Grouping of the n*k slots by expert: counts [E], exclusive offsets [E+1],
 * per-expert slot lists (token ascending) slot_token/slot_k [n*k], the
 * ascending list of experts with count > 0 and its length. */
void oracle_group(int n, int E, int k, const int32_t *topk_idx, int32_t *counts,
                  int32_t *offsets, int32_t *slot_token, int32_t *slot_k,
                  int32_t *unique, int32_t *U) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int t = 0; t < n; ++t)
        for (int j = 0; j < k; ++j) counts[topk_idx[(size_t)t * k + j]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int u = 0;
    for (int e = 0; e < E; ++e) {
        if (counts[e] > 0) unique[u++] = e;
        int pos = offsets[e];
        for (int t = 0; t < n; ++t)
            for (int j = 0; j < k; ++j)
                if (topk_idx[(size_t)t * k + j] == e) {
                    slot_token[pos] = t;
                    slot_k[pos] = j;
                    ++pos;
                }
    }
    *U = u;
}

/* Layer options beyond the default (SwiGLU, 4-bit down planes).
 * Activations (h = act(g, u)):
 *   ORACLE_ACT_SWIGLU         silu(g) * u, silu(z) = z / (1 + exp(-z))
 *   ORACLE_ACT_GEGLU          gelu(g) * u, gelu(z) = z * Phi(z) = z/2 (1 + erf(z / sqrt 2))
 *   ORACLE_ACT_GEGLU_TANH     gelu's tanh form: z/2 (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
 *   ORACLE_ACT_SWIGLU_CLAMPED silu(min(g, L)) * min(max(u, -L), L), L = limit
 * Sources: #1616 Implementation Notes names the GeGLU variant of the fused
 * kernel (gemma4); #1859 Problem / Background names the clamp stage of
 * deepseek_v4's limited SwiGLU. Neither page gives the formulas or the bounds:
 * GeGLU is read as the GLU with GELU (exact, and the tanh approximation as a
 * second kind), the clamp as bounding the gate from above and the up
 * projection on both sides at one limit L.
 * down_bits: 4 (uint32 words of eight codes) or 6 (#1616 Implementation Notes:
 * dots.llm1 has 4-bit gate/up with 6-bit down; the byte stream of
 * dequant6_at). */
typedef struct {
    int activation;
    float limit;
    int down_bits;
} oracle_options;

enum { ORACLE_ACT_SWIGLU = 0, ORACLE_ACT_GEGLU = 1, ORACLE_ACT_GEGLU_TANH = 2,
       ORACLE_ACT_SWIGLU_CLAMPED = 3 };

static float silu(float z) { return z / (1.0f + expf(-z)); }

static float glu_activation(const oracle_options *o, float g, float u) {
    switch (o->activation) {
        case ORACLE_ACT_GEGLU:
            return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f)) * u;
        case ORACLE_ACT_GEGLU_TANH: {
            float inner = 0.79788456080286536f * (g + 0.044715f * g * g * g);
            return 0.5f * g * (1.0f + tanhf(inner)) * u;
        }
        case ORACLE_ACT_SWIGLU_CLAMPED: {
            float gc = fminf(g, o->limit);
            float uc = fminf(fmaxf(u, -o->limit), o->limit);
            return silu(gc) * uc;
        }
        default:
            return silu(g) * u;
    }
}

/* One expert's gated MLP on one token (options as above):
 *   g_f = sum_d Wg[f,d] x[d],  u_f = sum_d Wu[f,d] x[d],
 *   h_f = act(g_f, u_f),       y_d = sum_f Wd[d,f] h_f.
 * Planes are those of a single expert (no E stride); dq holds uint32 words
 * (4-bit) or bytes (6-bit). h is caller scratch [F]. */
void oracle_expert_mlp_opt(int D, int F, const float *x,
                           const uint32_t *gq, const uint16_t *gs, const uint16_t *gb,
                           const uint32_t *uq, const uint16_t *us, const uint16_t *ub,
                           const void *dq, const uint16_t *ds, const uint16_t *db,
                           const oracle_options *opt, float *h, float *y) {
    for (int f = 0; f < F; ++f) {
        const uint32_t *gqr = gq + (size_t)f * (D / 8);
        const uint16_t *gsr = gs + (size_t)f * (D / ORACLE_GROUP);
        const uint16_t *gbr = gb + (size_t)f * (D / ORACLE_GROUP);
        const uint32_t *uqr = uq + (size_t)f * (D / 8);
        const uint16_t *usr = us + (size_t)f * (D / ORACLE_GROUP);
        const uint16_t *ubr = ub + (size_t)f * (D / ORACLE_GROUP);
        float g = 0.0f, u = 0.0f;
        for (int d = 0; d < D; ++d) {
            g = fmaf(dequant_at(gqr, gsr, gbr, d), x[d], g);
            u = fmaf(dequant_at(uqr, usr, ubr, d), x[d], u);
        }
        h[f] = glu_activation(opt, g, u);
    }
    for (int d = 0; d < D; ++d) {
        const uint16_t *dsr = ds + (size_t)d * (F / ORACLE_GROUP);
        const uint16_t *dbr = db + (size_t)d * (F / ORACLE_GROUP);
        float acc = 0.0f;
        if (opt->down_bits == 6) {
            const uint8_t *dqr = (const uint8_t *)dq + (size_t)d * (3 * F / 4);
            for (int f = 0; f < F; ++f) acc = fmaf(dequant6_at(dqr, dsr, dbr, f), h[f], acc);
        } else {
            const uint32_t *dqr = (const uint32_t *)dq + (size_t)d * (F / 8);
            for (int f = 0; f < F; ++f) acc = fmaf(dequant_at(dqr, dsr, dbr, f), h[f], acc);
        }
        y[d] = acc;
    }
}

static const oracle_options kDefaultOptions = {ORACLE_ACT_SWIGLU, 0.0f, 4};

/* The default layer: SwiGLU with 4-bit down planes. */
void oracle_expert_mlp(int D, int F, const float *x,
                       const uint32_t *gq, const uint16_t *gs, const uint16_t *gb,
                       const uint32_t *uq, const uint16_t *us, const uint16_t *ub,
                       const uint32_t *dq, const uint16_t *ds, const uint16_t *db,
                       float *h, float *y) {
    oracle_expert_mlp_opt(D, F, x, gq, gs, gb, uq, us, ub, dq, ds, db, &kDefaultOptions, h, y);
}

typedef struct {
    const uint32_t *gate_q; const uint16_t *gate_s; const uint16_t *gate_b;
    const uint32_t *up_q;   const uint16_t *up_s;   const uint16_t *up_b;
    const void *down_q;     const uint16_t *down_s; const uint16_t *down_b;  /* words or bytes */
} oracle_planes;

/* The whole decode step. Planes are stacked [E, ...] (see oracle_planes).
 * Outputs: routing (topk_idx, topk_w), grouping (counts, offsets, slot_token,
 * slot_k, unique, U), out_f32 [n,D] before rounding and, when out_bf16 is not
 * NULL, out rounded once to bf16 (round to nearest even). Returns 0, or -1 on
 * bad arguments or allocation failure. */
int oracle_moe_forward_opt(int E, int k, int D, int F, int n,
                           const float *x, const float *router_w, const float *router_bias,
                           const oracle_planes *pl, const oracle_options *opt,
                           int32_t *topk_idx, float *topk_w,
                           int32_t *counts, int32_t *offsets, int32_t *slot_token,
                           int32_t *slot_k, int32_t *unique, int32_t *U,
                           float *out_f32, uint16_t *out_bf16) {
    if (E < 1 || k < 1 || k > E || n < 1 || D % ORACLE_GROUP || F % ORACLE_GROUP) return -1;
    if (opt->down_bits != 4 && opt->down_bits != 6) return -1;
    oracle_route(n, E, D, k, x, router_w, router_bias, topk_idx, topk_w, NULL, NULL);
    oracle_group(n, E, k, topk_idx, counts, offsets, slot_token, slot_k, unique, U);

    const int S = n * k;
    float *y = (float *)malloc(sizeof(float) * (size_t)S * D);  /* y per slot, slot = t*k + j */
    if (!y) return -1;
    const size_t gstride = (size_t)F * (D / 8), gsstride = (size_t)F * (D / ORACLE_GROUP);
    /* bytes of one expert's down codes */
    const size_t dstride = (size_t)D * (opt->down_bits == 6 ? 3 * F / 4 : F / 2);
    const size_t dsstride = (size_t)D * (F / ORACLE_GROUP);
    int failed = 0;
#pragma omp parallel
    {
        float *h = (float *)malloc(sizeof(float) * (size_t)F);
        if (!h) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int slot = 0; slot < S; ++slot) {
            if (!h) continue;
            int t = slot / k, e = topk_idx[slot];
            oracle_expert_mlp_opt(D, F, x + (size_t)t * D,
                                  pl->gate_q + e * gstride, pl->gate_s + e * gsstride, pl->gate_b + e * gsstride,
                                  pl->up_q + e * gstride, pl->up_s + e * gsstride, pl->up_b + e * gsstride,
                                  (const uint8_t *)pl->down_q + e * dstride, pl->down_s + e * dsstride,
                                  pl->down_b + e * dsstride, opt, h, y + (size_t)slot * D);
        }
        free(h);
    }
    if (failed) { free(y); return -1; }
    /* combine: out[t] = sum_{j=0..k-1} w[t,j] * y[t,j] in rank order j */
    for (int t = 0; t < n; ++t)
        for (int d = 0; d < D; ++d) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j)
                acc = fmaf(topk_w[(size_t)t * k + j], y[((size_t)t * k + j) * D + d], acc);
            out_f32[(size_t)t * D + d] = acc;
        }
    if (out_bf16)
        for (size_t i = 0; i < (size_t)n * D; ++i) out_bf16[i] = bf16_round_rne(out_f32[i]);
    free(y);
    return 0;
}

/* The default layer (SwiGLU, 4-bit down planes). */
int oracle_moe_forward(int E, int k, int D, int F, int n,
                       const float *x, const float *router_w, const float *router_bias,
                       const oracle_planes *pl,
                       int32_t *topk_idx, float *topk_w,
                       int32_t *counts, int32_t *offsets, int32_t *slot_token,
                       int32_t *slot_k, int32_t *unique, int32_t *U,
                       float *out_f32, uint16_t *out_bf16) {
    return oracle_moe_forward_opt(E, k, D, F, n, x, router_w, router_bias, pl, &kDefaultOptions,
                                  topk_idx, topk_w, counts, offsets, slot_token, slot_k, unique, U,
                                  out_f32, out_bf16);
}

/* The single final rounding, exposed for tests. */
void oracle_round_bf16(const float *in, uint16_t *out, size_t count) {
    for (size_t i = 0; i < count; ++i) out[i] = bf16_round_rne(in[i]);
}
