/*
 * moe_oracle.c -- plain, slow CPU oracle for the MXFP4 mixture-of-experts FFN
 * layer with softmax top-K routing.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this file.  It shares no code, header, table or helper
 * with the CUDA library; it follows the plain definition of each step, in the
 * order the step is defined, with no blocking, fusion or reordering.
 *
 * Sources for what is computed (web pages on the method):
 *  - softmax-scored top-K selection at E=512, K=10: InferenceX, "MI355X
 *    Qwen3.5 SGLang" blog, section on the optimisations, PR #21421 (fused_topk);
 *  - the shared expert treated as one more routed expert (top-K + 1) in the
 *    same dispatch when its width equals the routed width: same blog,
 *    PR #20736; vLLM MiniMax M3 on MI355X, section "shared expert fusion";
 *  - grouping tokens by expert in fixed-height row tiles (32-row tiles):
 *    VibeSys Qwen3.5-397B on 4x MI300A, section "cheaper prefill and
 *    collectives";
 *  - MXFP4 expert weights dequantised inside the fused MoE kernel: VibeSys,
 *    section "baseline" and section "kernels and graph capture".
 * The pages do not print the bit format or the activation.  Readings used
 * here: E2M1 codes, two per byte (low nibble = even k), one E8M0 scale byte
 * per 32 consecutive k; gate rows [0, I) then up rows [I, 2I) in W13; SwiGLU
 * h = bf16(silu(g) * u); routing weights renormalised over the K selected;
 * lower expert index wins ties; the shared expert has id E and weight 1.
 *
 * Precision: fp32 throughout (softmax with expf, dot products accumulated in
 * fp32 with k ascending), the SwiGLU result rounded to bf16 (nearest even),
 * the combine accumulated in fp32 over slots in ascending order, the output
 * rounded to bf16.
 *
 * Parity pins (tests/test_oracle_*.py): exhaustive E2M1 x E8M0 decode against
 * the closed form; routing and FFN against double-precision brute force on
 * tiny shapes; closed forms (constant codes, one-hot codes); invariants
 * (renormalised weights sum to 1, permutation is a stable bijection, grouped
 * loop == per-token loop, shared-as-expert == routed + dense MLP, W2 scale +1
 * doubles the output exactly, token permutation equivariance).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_OK 0
#define REF_ERR_ARG 1
#define REF_ERR_NAN 2

/* ---------------------------------------------------------------- helpers */

static float ref_bits_to_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t ref_f32_to_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* bf16 stored as its 16-bit pattern; widening is exact. */
float moe_ref_bf16_to_f32(uint16_t h) { return ref_bits_to_f32((uint32_t)h << 16); }

/* fp32 -> bf16, IEEE round to nearest, ties to even; NaN stays NaN. */
uint16_t moe_ref_f32_to_bf16(float f) {
    uint32_t u = ref_f32_to_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

/* E2M1 (1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit): codes 0..7
 * are 0, 0.5, 1, 1.5, 2, 3, 4, 6; codes 8..15 are the same values negated
 * (code 8 is -0). */
static const float ref_e2m1_value[16] = {0.0f,  0.5f,  1.0f,  1.5f,  2.0f,  3.0f,  4.0f,  6.0f,
                                         -0.0f, -0.5f, -1.0f, -1.5f, -2.0f, -3.0f, -4.0f, -6.0f};

float moe_ref_e2m1(int code) { return ref_e2m1_value[code & 15]; }

/* E8M0 scale byte s encodes 2^(s-127); 255 encodes NaN. */
float moe_ref_e8m0(int s) {
    if (s == 255) return NAN;
    return ldexpf(1.0f, s - 127);
}

/* One row of MXFP4 weights decoded to fp32: element k of the row is
 * E2M1(code_k) * 2^(s_{k/32} - 127), where code_k is the low nibble of byte
 * k/2 when k is even and the high nibble when k is odd. */
static void ref_decode_row(const uint8_t* codes_row, const uint8_t* scales_row, int len, float* out) {
    for (int g = 0; g < len / 32; ++g) {
        float scale = moe_ref_e8m0(scales_row[g]);
        for (int k = 32 * g; k < 32 * g + 32; ++k) {
            int byte = codes_row[k / 2];
            int code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            out[k] = moe_ref_e2m1(code) * scale;
        }
    }
}

double moe_ref_mxfp4_value(int code, int scale) {
    return (double)(moe_ref_e2m1(code) * moe_ref_e8m0(scale));
}

float moe_ref_silu(float g) { return g / (1.0f + expf(-g)); }

/* ----------------------------------------------------------------- route */

/* Softmax over all E logits of each token, then the K experts with the
 * largest logits (descending; equal logits -> lower index first), then their
 * probabilities renormalised to sum to one.  With the shared expert, slot K
 * holds expert E with weight 1.  Selecting on logits is the same as selecting
 * on probabilities (softmax is monotone) but free of ties created by rounding
 * in exp. */
int moe_ref_route(const float* logits, const float* shared_w, int T, int E, int K,
                  int with_shared, int renormalize, int32_t* topk_ids, float* topk_w) {
    if (T < 0 || E < 1 || K < 1 || K > E) return REF_ERR_ARG;
    int Kt = K + (with_shared ? 1 : 0);
    float* p = (float*)malloc(sizeof(float) * (size_t)E);
    int* taken = (int*)malloc(sizeof(int) * (size_t)E);
    if (!p || !taken) { free(p); free(taken); return REF_ERR_ARG; }
    int status = REF_OK;
    for (int t = 0; t < T && status == REF_OK; ++t) {
        const float* l = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            if (isnan(l[e])) status = REF_ERR_NAN;
        if (status != REF_OK) break;
        /* softmax */
        float m = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > m) m = l[e];
        float z = 0.0f;
        for (int e = 0; e < E; ++e) {
            p[e] = expf(l[e] - m);
            z += p[e];
        }
        for (int e = 0; e < E; ++e) p[e] = p[e] / z;
        /* top-K by logit: K rounds of "largest remaining, lowest index on ties" */
        for (int e = 0; e < E; ++e) taken[e] = 0;
        int32_t* ids = topk_ids + (size_t)t * Kt;
        float* w = topk_w + (size_t)t * Kt;
        for (int k = 0; k < K; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict: keeps the lower index on ties */
            }
            taken[best] = 1;
            ids[k] = best;
        }
        /* renormalise over the selected experts, in slot order */
        float s = 0.0f;
        for (int k = 0; k < K; ++k) s += p[ids[k]];
        for (int k = 0; k < K; ++k) w[k] = renormalize ? p[ids[k]] / s : p[ids[k]];
        if (with_shared) {
            ids[K] = E;
            w[K] = shared_w ? shared_w[t] : 1.0f; /* caller-supplied weight, e.g. a sigmoid gate */
        }
    }
    free(p);
    free(taken);
    return status;
}

/* --------------------------------------------------------------- permute */

int64_t moe_ref_capacity(int T, int Kt, int Et, int tile_m) {
    return (int64_t)T * Kt + (int64_t)Et * (tile_m - 1);
}

/* Counting sort of the T*Kt (token, slot) pairs by expert.  Pair q = t*Kt + j
 * goes to bucket topk_ids[q]; buckets keep pairs in increasing q.  Bucket e
 * starts at offsets[e] = sum over e' < e of count(e') rounded up to tile_m.
 * Unused positions up to the capacity hold -1.  inv[q] is the position of q.
 * Tile i covers positions [i*tile_m, (i+1)*tile_m) and tile_expert[i] is the
 * bucket it lies in; tiles from num_tiles up to max_tiles hold -1. */
int moe_ref_permute(const int32_t* topk_ids, int T, int Kt, int Et, int tile_m,
                    int32_t* sorted_pairs, int32_t* offsets, int32_t* inv,
                    int32_t* tile_expert, int32_t* num_tiles) {
    if (T < 0 || Kt < 1 || Et < 1 || tile_m < 1) return REF_ERR_ARG;
    int64_t P = (int64_t)T * Kt;
    int64_t cap = moe_ref_capacity(T, Kt, Et, tile_m);
    int64_t max_tiles = cap / tile_m;
    int64_t* count = (int64_t*)calloc((size_t)Et, sizeof(int64_t));
    int64_t* cursor = (int64_t*)calloc((size_t)Et, sizeof(int64_t));
    if (!count || !cursor) { free(count); free(cursor); return REF_ERR_ARG; }
    for (int64_t q = 0; q < P; ++q) {
        int e = topk_ids[q];
        if (e < 0 || e >= Et) { free(count); free(cursor); return REF_ERR_ARG; }
        count[e] += 1;
    }
    int64_t acc = 0;
    for (int e = 0; e < Et; ++e) {
        offsets[e] = (int32_t)acc;
        acc += (count[e] + tile_m - 1) / tile_m * tile_m;
    }
    offsets[Et] = (int32_t)acc;
    for (int64_t i = 0; i < cap; ++i) sorted_pairs[i] = -1;
    for (int64_t q = 0; q < P; ++q) {
        int e = topk_ids[q];
        int64_t pos = offsets[e] + cursor[e];
        cursor[e] += 1;
        sorted_pairs[pos] = (int32_t)q;
        inv[q] = (int32_t)pos;
    }
    int64_t nt = acc / tile_m;
    for (int64_t i = 0; i < max_tiles; ++i) tile_expert[i] = -1;
    for (int64_t i = 0; i < nt; ++i) {
        int64_t row = i * tile_m;
        int e = 0;
        while (!(offsets[e] <= row && row < offsets[e + 1])) ++e;
        tile_expert[i] = e;
    }
    *num_tiles = (int32_t)nt;
    free(count);
    free(cursor);
    return REF_OK;
}

/* ------------------------------------------------------------------- ffn */

/* One expert applied to one token:
 *   g_n = sum_k W13[n][k] x[k],  u_n = sum_k W13[I+n][k] x[k]   (fp32, k ascending)
 *   h_n = bf16(silu(g_n) * u_n)
 *   y_m = sum_n W2[m][n] h_n                                     (fp32, n ascending)
 * h_out (optional) receives the bf16 h as fp32 values. */
static void ref_expert_forward(const uint16_t* x_row, const uint8_t* w13, const uint8_t* s13,
                               const uint8_t* w2, const uint8_t* s2, int H, int I,
                               float* h, float* y) {
    float* xf = (float*)malloc(sizeof(float) * (size_t)H);
    float* wg = (float*)malloc(sizeof(float) * (size_t)H);
    float* wu = (float*)malloc(sizeof(float) * (size_t)H);
    float* wd = (float*)malloc(sizeof(float) * (size_t)I);
    for (int k = 0; k < H; ++k) xf[k] = moe_ref_bf16_to_f32(x_row[k]);
    for (int n = 0; n < I; ++n) {
        ref_decode_row(w13 + (size_t)n * (H / 2), s13 + (size_t)n * (H / 32), H, wg);
        ref_decode_row(w13 + (size_t)(I + n) * (H / 2), s13 + (size_t)(I + n) * (H / 32), H, wu);
        float g = 0.0f, u = 0.0f;
        for (int k = 0; k < H; ++k) {
            g += wg[k] * xf[k];
            u += wu[k] * xf[k];
        }
        h[n] = moe_ref_bf16_to_f32(moe_ref_f32_to_bf16(moe_ref_silu(g) * u));
    }
    for (int m = 0; m < H; ++m) {
        ref_decode_row(w2 + (size_t)m * (I / 2), s2 + (size_t)m * (I / 32), I, wd);
        float acc = 0.0f;
        for (int n = 0; n < I; ++n) acc += wd[n] * h[n];
        y[m] = acc;
    }
    free(xf);
    free(wg);
    free(wu);
    free(wd);
}

static int ref_ffn_args_ok(int T, int H, int I, int Et, int Kt) {
    return T >= 0 && H > 0 && I > 0 && Et > 0 && Kt > 0 && H % 32 == 0 && I % 32 == 0;
}

/* Per-token loop (the definition): for each requested token t, for each slot
 * j ascending, acc += w[t][j] * expert_{ids[t][j]}(x_t); out_t = bf16(acc).
 * tokens[i] selects which token row i of the outputs holds (NULL: all T in
 * order, n_tokens = T).  out_f32 (optional) receives acc before rounding.
 * n_threads > 1 spreads tokens over OpenMP threads; the per-token order of
 * operations does not change. */
int moe_ref_ffn(const uint16_t* x, const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                const uint8_t* s2, const int32_t* topk_ids, const float* topk_w, int T, int H,
                int I, int Et, int Kt, const int32_t* tokens, int n_tokens, uint16_t* out,
                float* out_f32, int n_threads) {
    if (!ref_ffn_args_ok(T, H, I, Et, Kt) || n_tokens < 0) return REF_ERR_ARG;
    if (!tokens && n_tokens != T) return REF_ERR_ARG;
    for (int i = 0; i < n_tokens; ++i) {
        int t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) return REF_ERR_ARG;
        for (int j = 0; j < Kt; ++j) {
            int e = topk_ids[(size_t)t * Kt + j];
            if (e < 0 || e >= Et) return REF_ERR_ARG;
        }
    }
    size_t w13_e = (size_t)2 * I * (H / 2), s13_e = (size_t)2 * I * (H / 32);
    size_t w2_e = (size_t)H * (I / 2), s2_e = (size_t)H * (I / 32);
#ifdef _OPENMP
    if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int i = 0; i < n_tokens; ++i) {
        int t = tokens ? tokens[i] : i;
        float* h = (float*)malloc(sizeof(float) * (size_t)I);
        float* y = (float*)malloc(sizeof(float) * (size_t)H);
        float* acc = (float*)malloc(sizeof(float) * (size_t)H);
        for (int m = 0; m < H; ++m) acc[m] = 0.0f;
        for (int j = 0; j < Kt; ++j) {
            int e = topk_ids[(size_t)t * Kt + j];
            float wj = topk_w[(size_t)t * Kt + j];
            ref_expert_forward(x + (size_t)t * H, w13 + e * w13_e, s13 + e * s13_e, w2 + e * w2_e,
                               s2 + e * s2_e, H, I, h, y);
            for (int m = 0; m < H; ++m) acc[m] += wj * y[m];
        }
        for (int m = 0; m < H; ++m) {
            out[(size_t)i * H + m] = moe_ref_f32_to_bf16(acc[m]);
            if (out_f32) out_f32[(size_t)i * H + m] = acc[m];
        }
        free(h);
        free(y);
        free(acc);
    }
    return REF_OK;
}

/* Expert-major variant driven by the permutation: walk the buckets in expert
 * order, compute every pair's weighted expert output once, then combine each
 * token's slots in ascending order.  Same per-pair arithmetic as moe_ref_ffn,
 * so the results must agree bit for bit (an invariant the tests check). */
int moe_ref_ffn_grouped(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                        const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                        const int32_t* sorted_pairs, const int32_t* offsets, int T, int H, int I,
                        int Et, int Kt, uint16_t* out) {
    if (!ref_ffn_args_ok(T, H, I, Et, Kt)) return REF_ERR_ARG;
    size_t P = (size_t)T * Kt;
    float* ypair = (float*)malloc(sizeof(float) * P * (size_t)H);
    float* h = (float*)malloc(sizeof(float) * (size_t)I);
    float* y = (float*)malloc(sizeof(float) * (size_t)H);
    size_t w13_e = (size_t)2 * I * (H / 2), s13_e = (size_t)2 * I * (H / 32);
    size_t w2_e = (size_t)H * (I / 2), s2_e = (size_t)H * (I / 32);
    for (int e = 0; e < Et; ++e) {
        for (int32_t pos = offsets[e]; pos < offsets[e + 1]; ++pos) {
            int32_t q = sorted_pairs[pos];
            if (q < 0) continue;
            int t = q / Kt;
            ref_expert_forward(x + (size_t)t * H, w13 + e * w13_e, s13 + e * s13_e,
                               w2 + e * w2_e, s2 + e * s2_e, H, I, h, y);
            for (int m = 0; m < H; ++m) ypair[(size_t)q * H + m] = topk_w[q] * y[m];
        }
    }
    for (int t = 0; t < T; ++t) {
        for (int m = 0; m < H; ++m) {
            float acc = 0.0f;
            for (int j = 0; j < Kt; ++j) acc += ypair[((size_t)t * Kt + j) * H + m];
            out[(size_t)t * H + m] = moe_ref_f32_to_bf16(acc);
        }
    }
    free(ypair);
    free(h);
    free(y);
    return REF_OK;
}

/* ------------------------------------------- MXFP4-quantised activations */

/* E2M1 code (0..15) of v rounded to the nearest E2M1 value: the magnitude
 * goes to the nearest of the eight non-negative values (equal distance: the
 * even code, i.e. the value whose last mantissa bit is 0), magnitudes above
 * 6 to 6 (saturation); the sign bit of v is kept, so a negative v that rounds
 * to zero gives code 8 (-0).  v must be finite. */
static int ref_e2m1_round(double v) {
    double a = fabs(v);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(a - (double)ref_e2m1_value[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) != 0)) {
            best = c;
            best_d = d;
        }
    }
    return best | (signbit(v) ? 8 : 0);
}

int moe_ref_e2m1_round(double v) { return ref_e2m1_round(v); }

/* MXFP4 quantisation of n values (n a multiple of 32), following the OCP
 * Microscaling Formats (MX) v1.0 conversion: for each block of 32 consecutive
 * values, amax = the largest magnitude; the shared exponent is
 * e = floor(log2(amax)) - 2, where 2 is the exponent of E2M1's largest value
 * (6 = 1.5 * 2^2), clamped to the E8M0 range [-127, 127]; the block's scale
 * byte is e + 127 and element k's code is ref_e2m1_round(v_k / 2^e).  A block
 * whose values are all zero gets scale byte 0 and zero codes.  Codes are
 * packed two per byte, element 2i in the low nibble.  The pages fuse this
 * quantisation into the activation kernel that feeds an MXFP4 x MXFP4 GEMM
 * (OpenRelay, "Gemma 4 31B from B200 to MI355X": section "optimisation 4",
 * the fused GELU + up projection + MXFP4 quantisation kernel; section "how
 * far from the ceiling", matmuls measured against the MXFP4 peak); they do
 * not print the rounding, so the OCP rule is the reading taken here.
 * Returns REF_ERR_NAN on a non-finite value. */
int moe_ref_quantize_mxfp4(const float* v, int n, uint8_t* codes, uint8_t* scales) {
    if (n < 0 || n % 32 != 0) return REF_ERR_ARG;
    for (int b = 0; b < n / 32; ++b) {
        const float* blk = v + 32 * b;
        double amax = 0.0;
        for (int k = 0; k < 32; ++k) {
            if (!isfinite(blk[k])) return REF_ERR_NAN;
            if (fabs((double)blk[k]) > amax) amax = fabs((double)blk[k]);
        }
        int e;
        if (amax == 0.0) {
            e = -127;
        } else {
            int ex;
            frexp(amax, &ex); /* amax = m * 2^ex, m in [0.5, 1): floor(log2(amax)) = ex - 1 */
            e = ex - 1 - 2;
            if (e < -127) e = -127;
            if (e > 127) e = 127;
        }
        scales[b] = (uint8_t)(amax == 0.0 ? 0 : e + 127);
        for (int k = 0; k < 32; k += 2) {
            int c0 = amax == 0.0 ? 0 : ref_e2m1_round(ldexp((double)blk[k], -e));
            int c1 = amax == 0.0 ? 0 : ref_e2m1_round(ldexp((double)blk[k + 1], -e));
            codes[(32 * b + k) / 2] = (uint8_t)(c0 | (c1 << 4));
        }
    }
    return REF_OK;
}

/* One (token, expert) pair with MXFP4-quantised activations:
 *   xq  = dequantise(quantise_mxfp4(x))                 (blocks of 32 along H)
 *   g_n = sum_k W13[n][k] xq[k],  u_n = sum_k W13[I+n][k] xq[k]  (fp32, k ascending)
 *   a_n = silu(g_n) * u_n                                (fp32, not rounded)
 *   hq  = dequantise(quantise_mxfp4(a))                  (blocks of 32 along I)
 *   y_m = sum_n W2[m][n] hq[n]                           (fp32, n ascending)
 * a (the pre-quantisation SwiGLU output), hcodes and hscales receive the
 * intermediate values. */
static int ref_expert_forward_mxfp4(const float* xq, const uint8_t* w13, const uint8_t* s13,
                                    const uint8_t* w2, const uint8_t* s2, int H, int I,
                                    float* a, uint8_t* hcodes, uint8_t* hscales, float* y) {
    float* wg = (float*)malloc(sizeof(float) * (size_t)H);
    float* wu = (float*)malloc(sizeof(float) * (size_t)H);
    float* wd = (float*)malloc(sizeof(float) * (size_t)I);
    float* hq = (float*)malloc(sizeof(float) * (size_t)I);
    for (int n = 0; n < I; ++n) {
        ref_decode_row(w13 + (size_t)n * (H / 2), s13 + (size_t)n * (H / 32), H, wg);
        ref_decode_row(w13 + (size_t)(I + n) * (H / 2), s13 + (size_t)(I + n) * (H / 32), H, wu);
        float g = 0.0f, u = 0.0f;
        for (int k = 0; k < H; ++k) {
            g += wg[k] * xq[k];
            u += wu[k] * xq[k];
        }
        a[n] = moe_ref_silu(g) * u;
    }
    int rc = moe_ref_quantize_mxfp4(a, I, hcodes, hscales);
    if (rc == REF_OK) {
        ref_decode_row(hcodes, hscales, I, hq);
        for (int m = 0; m < H; ++m) {
            ref_decode_row(w2 + (size_t)m * (I / 2), s2 + (size_t)m * (I / 32), I, wd);
            float acc = 0.0f;
            for (int n = 0; n < I; ++n) acc += wd[n] * hq[n];
            y[m] = acc;
        }
    }
    free(wg);
    free(wu);
    free(wd);
    free(hq);
    return rc;
}

/* The layer with MXFP4-quantised activations, per-token loop: like moe_ref_ffn
 * with each expert evaluated by ref_expert_forward_mxfp4 on the token's
 * quantised row.  For the requested tokens (tokens / n_tokens as in
 * moe_ref_ffn), the optional outputs receive per pair (row i * Kt + j): a_out
 * [.., I] the SwiGLU output before quantisation, hcodes_out [.., I/2] and
 * hscales_out [.., I/32] its MXFP4 encoding.  H % 32 == 0, I % 32 == 0. */
int moe_ref_ffn_mxfp4act(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                         const uint8_t* w2, const uint8_t* s2, const int32_t* topk_ids,
                         const float* topk_w, int T, int H, int I, int Et, int Kt,
                         const int32_t* tokens, int n_tokens, uint16_t* out, float* out_f32,
                         float* a_out, uint8_t* hcodes_out, uint8_t* hscales_out, int n_threads) {
    if (!ref_ffn_args_ok(T, H, I, Et, Kt) || n_tokens < 0) return REF_ERR_ARG;
    if (!tokens && n_tokens != T) return REF_ERR_ARG;
    for (int i = 0; i < n_tokens; ++i) {
        int t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) return REF_ERR_ARG;
        for (int j = 0; j < Kt; ++j) {
            int e = topk_ids[(size_t)t * Kt + j];
            if (e < 0 || e >= Et) return REF_ERR_ARG;
        }
    }
    size_t w13_e = (size_t)2 * I * (H / 2), s13_e = (size_t)2 * I * (H / 32);
    size_t w2_e = (size_t)H * (I / 2), s2_e = (size_t)H * (I / 32);
    int status = REF_OK;
#ifdef _OPENMP
    if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int i = 0; i < n_tokens; ++i) {
        int t = tokens ? tokens[i] : i;
        float* xf = (float*)malloc(sizeof(float) * (size_t)H);
        float* xq = (float*)malloc(sizeof(float) * (size_t)H);
        uint8_t* xc = (uint8_t*)malloc((size_t)H / 2);
        uint8_t* xs = (uint8_t*)malloc((size_t)H / 32);
        float* a = (float*)malloc(sizeof(float) * (size_t)I);
        uint8_t* hc = (uint8_t*)malloc((size_t)I / 2);
        uint8_t* hs = (uint8_t*)malloc((size_t)I / 32);
        float* y = (float*)malloc(sizeof(float) * (size_t)H);
        float* acc = (float*)malloc(sizeof(float) * (size_t)H);
        for (int k = 0; k < H; ++k) xf[k] = moe_ref_bf16_to_f32(x[(size_t)t * H + k]);
        int rc = moe_ref_quantize_mxfp4(xf, H, xc, xs);
        if (rc == REF_OK) ref_decode_row(xc, xs, H, xq);
        for (int m = 0; m < H; ++m) acc[m] = 0.0f;
        for (int j = 0; j < Kt && rc == REF_OK; ++j) {
            int e = topk_ids[(size_t)t * Kt + j];
            float wj = topk_w[(size_t)t * Kt + j];
            rc = ref_expert_forward_mxfp4(xq, w13 + e * w13_e, s13 + e * s13_e, w2 + e * w2_e,
                                          s2 + e * s2_e, H, I, a, hc, hs, y);
            if (rc != REF_OK) break;
            size_t r = (size_t)i * Kt + j;
            if (a_out) memcpy(a_out + r * I, a, sizeof(float) * (size_t)I);
            if (hcodes_out) memcpy(hcodes_out + r * (I / 2), hc, (size_t)I / 2);
            if (hscales_out) memcpy(hscales_out + r * (I / 32), hs, (size_t)I / 32);
            for (int m = 0; m < H; ++m) acc[m] += wj * y[m];
        }
        if (rc != REF_OK) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = rc;
        }
        for (int m = 0; m < H; ++m) {
            out[(size_t)i * H + m] = moe_ref_f32_to_bf16(acc[m]);
            if (out_f32) out_f32[(size_t)i * H + m] = acc[m];
        }
        free(xf);
        free(xq);
        free(xc);
        free(xs);
        free(a);
        free(hc);
        free(hs);
        free(y);
        free(acc);
    }
    return status;
}

int moe_ref_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
