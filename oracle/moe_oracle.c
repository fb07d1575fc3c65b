/*
 * moe_oracle.c -- plain, slow fp64 CPU oracle for the forward pass of one
 * Mixture-of-Experts (MoE) layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file (through oracle/__init__.py).
 * The CUDA library never includes, links or calls it, and it shares no source
 * with the CUDA library: no headers, helpers, tables or constants.
 *
 * What it computes, step by step (each function cites the passage it follows):
 *   1. router: logits = x . Wg^T (+ optional per-expert logit bias), a softmax
 *      over all experts, top-k by logit with ties to the lower expert id, and
 *      optional renormalisation of the k probabilities;
 *   2. expert -> expert-slot map (identity, or a replica table);
 *   3. optional expert-parallel local-range mask and remap;
 *   4. per-slot counts, exclusive-scan offsets, and the stable permutation of
 *      (token, k) pairs grouped by slot;
 *   5. per selected expert a gated MLP (SwiGLU) with the intermediate rounded
 *      to bf16, and one routing-weighted sum over the k experts per token, plus
 *      optional shared experts (optionally scaled by a sigmoid gate).
 *
 * Arithmetic: every input is bf16 or fp32; products of a bf16 with a bf16 or
 * fp32 value are exact in fp64, sums run in fp64 in ascending index order, and
 * exp() is the C library's double-precision exp.  The one deliberate rounding
 * is the SwiGLU intermediate h, rounded to bf16 (round to nearest, ties to
 * even) as the GPU path also does.  Build with -ffp-contract=off so x86 and Arm
 * hosts give bit-identical results.
 *
 * Parity pins: tests/test_oracle_pins.py checks every function here against
 * closed forms, brute force, invariants and independent library routines.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_NONLOCAL_SKIP 0
#define ORACLE_NONLOCAL_MOD 1

/* ------------------------------------------------------------------------- */
/* bf16 <-> double                                                            */
/* ------------------------------------------------------------------------- */

/* A bf16 value is the upper 16 bits of an IEEE binary32 value. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even (8 significant bits,
 * binary32 exponent range, gradual underflow with spacing 2^-133, overflow to
 * infinity).  Done on the value itself: scale by a power of two so the last
 * kept bit has weight 1, round to an integer with nearbyint() under the
 * default round-to-nearest-even mode, scale back. */
uint16_t oracle_f64_to_bf16(double v)
{
    if (isnan(v)) return (uint16_t)0x7FC0u;
    uint16_t sign = signbit(v) ? (uint16_t)0x8000u : (uint16_t)0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int e;
    (void)frexp(a, &e);            /* a = m * 2^e with m in [0.5, 1) */
    int lsb = (e - 1) - 7;         /* weight of the 8th significant bit */
    if (lsb < -133) lsb = -133;    /* bf16 subnormal spacing */
    double q = ldexp(a, -lsb);     /* exact */
    double r = nearbyint(q);       /* ties to even */
    double res = ldexp(r, lsb);    /* exact */
    const double bf16_max = 3.3895313892515355e38; /* (2 - 2^-7) * 2^127 */
    if (res > bf16_max) return (uint16_t)(sign | 0x7F80u);
    float f = (float)res; /* exact: res has <= 8 significant bits in range */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFFu));
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 weights with one fp32 scale per row                               */
/* ------------------------------------------------------------------------- */

/* FP8 expert weights (TensorRT-LLM AutoDeploy MoE PR #10985, review of
 * torch_moe.py: the MoE ops have FP8 and NVFP4 paths).  The pages give no
 * format; the reading taken is the plainest one: OCP E4M3 ("fn": sign, 4
 * exponent bits with bias 7, 3 mantissa bits, no infinities, 0x7F / 0xFF NaN,
 * largest finite 448, subnormal spacing 2^-9) with one fp32 scale per output
 * row, W[r][c] = scale[r] * e4m3(q[r][c]). */
double oracle_e4m3_to_f64(uint8_t q)
{
    const int sgn = q >> 7, e = (q >> 3) & 0xF, m = q & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* Nearest E4M3 value, ties to even, finite results saturated at +-448
 * (as a saturating conversion does); NaN -> 0x7F. */
uint8_t oracle_f64_to_e4m3(double v)
{
    if (isnan(v)) return 0x7F;
    const uint8_t sgn = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a == 0.0) return sgn;
    int e;
    (void)frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
    int lsb = (e - 1) - 3;         /* weight of the 4th significant bit */
    if (lsb < -9) lsb = -9;        /* subnormal spacing */
    double r = ldexp(nearbyint(ldexp(a, -lsb)), lsb);  /* ties to even */
    if (r > 448.0) r = 448.0;
    if (r < ldexp(1.0, -6)) {      /* subnormal (or zero): m * 2^-9 */
        return (uint8_t)(sgn | (uint8_t)ldexp(r, 9));
    }
    (void)frexp(r, &e);
    const int E = e - 1 + 7;       /* r = (1 + m/8) * 2^(e-1) */
    const int m = (int)(ldexp(r, -(e - 1)) * 8.0) - 8;
    return (uint8_t)(sgn | (uint8_t)(E << 3) | (uint8_t)m);
}

/* Row-wise quantisation of a bf16 matrix [rows, K]: scale = amax / 448 (an
 * IEEE binary32 division), q = e4m3(w / scale) with the division again in
 * binary32; an all-zero row gets scale 0 and q = 0. */
void oracle_quantize_fp8_rows(const uint16_t *w, int64_t rows, int K, uint8_t *q, float *scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *wr = w + (size_t)r * (size_t)K;
        float amax = 0.0f;
        for (int c = 0; c < K; ++c) {
            const float f = (float)oracle_bf16_to_f64(wr[c]);
            if (fabsf(f) > amax) amax = fabsf(f);
        }
        volatile float sc = amax / 448.0f;
        scale[r] = sc;
        for (int c = 0; c < K; ++c) {
            if (sc == 0.0f) {
                q[(size_t)r * (size_t)K + (size_t)c] = 0;
                continue;
            }
            volatile float v = (float)oracle_bf16_to_f64(wr[c]) / sc;
            q[(size_t)r * (size_t)K + (size_t)c] = oracle_f64_to_e4m3((double)v);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* NVFP4 values: E2M1 elements, an E4M3 scale per 16 consecutive elements of a */
/* row, and an fp32 scale per row                                             */
/* ------------------------------------------------------------------------- */

/* E2M1 code (bit 3 sign, bits 2-1 exponent with bias 1, bit 0 mantissa): the
 * magnitudes 0, 0.5 (exponent field 0: m * 0.5), 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_to_f64(uint8_t q)
{
    const int sgn = (q >> 3) & 1, e = (q >> 1) & 3, m = q & 1;
    const double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sgn ? -v : v;
}

/* Nearest E2M1 value, ties to even (the code whose mantissa bit is 0), finite
 * results saturated at +-6; returns the 4-bit code.  Inputs are finite. */
uint8_t oracle_f64_to_e2m1(double v)
{
    const uint8_t sgn = signbit(v) ? 8 : 0;
    const double a = fabs(v);
    if (a == 0.0) return sgn;
    int e;
    (void)frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
    int lsb = (e - 1) - 1;         /* weight of the 2nd significant bit */
    if (lsb < -1) lsb = -1;        /* subnormal spacing 0.5 */
    double r = ldexp(nearbyint(ldexp(a, -lsb)), lsb);  /* ties to even */
    if (r > 6.0) r = 6.0;
    if (r < 1.0) return (uint8_t)(sgn | (uint8_t)(r * 2.0));  /* 0 or 0.5 */
    (void)frexp(r, &e);
    const int E = e;               /* r = (1 + m/2) * 2^(e-1), exponent field e - 1 + 1 */
    const int m = (int)(ldexp(r, -(e - 1)) * 2.0) - 2;
    return (uint8_t)(sgn | (uint8_t)(E << 1) | (uint8_t)m);
}

/* NVFP4 quantisation of one bf16 row [K], K a multiple of 16.  The pages name
 * NVFP4 expert weights (TensorRT-LLM PR #10985, review of torch_moe.py, which
 * names the FP8 and NVFP4 paths of the MoE ops) and define no encoding.
 * Reading: the row's fp32 scale is s = amax / (6 * 448), one binary32 division
 * (6 * 448 = 2688 is exact); each block of 16 consecutive elements gets the
 * E4M3 scale sb = e4m3(amax_b / (6 * s)), the product 6 * s and the division in
 * binary32, rounded to E4M3 to nearest with ties to even and saturated at 448;
 * each element q = e2m1(v / (sb * s)), the product sb * s and the division in
 * binary32.  The value is e2m1(q) * sb * s.  An all-zero row gets s = 0, zero
 * block scales and zero codes; a block whose scale rounds to 0 gets zero codes.
 * q holds one code per element (0..15); sb one E4M3 byte per block.
 *
 * pow2 (activations): the row scale is instead the power of two s = 2^e, e the
 * smallest integer >= -126 with amax <= 2688 * 2^e (an all-zero row gets
 * 2^-126), for the reason E4M3 activations use one: the GPU's bf16 rows can
 * differ from the oracle's in a rare last bit, and a scale set by amax itself
 * would then move every block scale and code of the row. */
void oracle_quantize_nvfp4_row(const uint16_t *v, int K, int pow2, uint8_t *q, uint8_t *sb, float *scale)
{
    float amax = 0.0f;
    for (int c = 0; c < K; ++c) {
        const float f = fabsf((float)oracle_bf16_to_f64(v[c]));
        if (f > amax) amax = f;
    }
    volatile float s = amax / 2688.0f;
    if (pow2) {
        int e = -126;
        while ((double)amax > ldexp(2688.0, e)) ++e;
        s = (float)ldexp(1.0, e);
    }
    *scale = s;
    for (int b = 0; b < K / 16; ++b) {
        float bmax = 0.0f;
        for (int c = 16 * b; c < 16 * b + 16; ++c) {
            const float f = fabsf((float)oracle_bf16_to_f64(v[c]));
            if (f > bmax) bmax = f;
        }
        uint8_t code = 0;
        if (s != 0.0f) {
            volatile float six_s = 6.0f * s;
            volatile float d = bmax / six_s;
            code = oracle_f64_to_e4m3((double)d);
        }
        sb[b] = code;
        const float sbv = (float)oracle_e4m3_to_f64(code);
        volatile float denom = sbv * s;
        for (int c = 16 * b; c < 16 * b + 16; ++c) {
            if (denom == 0.0f) {
                q[c] = 0;
                continue;
            }
            volatile float x = (float)oracle_bf16_to_f64(v[c]) / denom;
            q[c] = oracle_f64_to_e2m1((double)x);
        }
    }
}

void oracle_quantize_nvfp4_rows(const uint16_t *v, int64_t rows, int K, int pow2, uint8_t *q, uint8_t *sb,
                                float *scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        oracle_quantize_nvfp4_row(v + (size_t)r * (size_t)K, K, pow2, q + (size_t)r * (size_t)K,
                                  sb + (size_t)r * (size_t)(K / 16), scale + r);
}

/* A weight matrix of the layer: bf16 values, E4M3 bytes with row scales, or
 * (sb given) NVFP4 codes with block and row scales. */
typedef struct {
    const uint16_t *bf;
    const uint8_t *q;
    const float *s;
    size_t K;
    const uint8_t *sb;
} oracle_wmat;

static double wget(const oracle_wmat *m, size_t row, size_t col)
{
    const size_t i = row * m->K + col;
    if (m->sb)
        return (double)m->s[row] * oracle_e4m3_to_f64(m->sb[row * (m->K / 16) + col / 16]) *
               oracle_e2m1_to_f64(m->q[i]);
    return m->q ? (double)m->s[row] * oracle_e4m3_to_f64(m->q[i]) : oracle_bf16_to_f64(m->bf[i]);
}

/* ------------------------------------------------------------------------- */
/* 1. Router                                                                  */
/* ------------------------------------------------------------------------- */

/* Router for tokens t in [0, T): gate logits, softmax over all E experts, top-k
 * by logit (ties to the lower expert id), optional renormalisation.
 *
 * Follows the vLLM EP FusedMoE patch (ep_fused_moe_patch.py), module docstring
 * "EP expert dispatch": top-k routing produces global expert ids, identical on
 * every rank; and its patched FusedMoE __init__ (renormalize=True default,
 * routing over the global expert count).  Softmax over all experts comes
 * first, then top-k ("softmax-then-top-k with renorm").  Selection is on the
 * logits: softmax is strictly increasing in the logit, so the order is the
 * same, and ties between distinct logits cannot be created by rounding of
 * probabilities.
 *
 *   x       [T, H] bf16 bits      Wg [E, H] fp32      bias [E] fp32 or NULL
 *   ids     [T, k] int32 out      (descending logit, ties to lower id)
 *   w       [T, k] double out     (p_e, or p_e / sum of the k selected p)
 *   logits  [T, E] double out, or NULL
 */
void oracle_route_grouped(const uint16_t *x, const float *Wg, const float *bias,
                          int64_t T, int H, int E, int k, int renorm, int n_group, int topk_group,
                          int32_t *ids, double *w, double *logits);

void oracle_route(const uint16_t *x, const float *Wg, const float *bias,
                  int64_t T, int H, int E, int k, int renorm,
                  int32_t *ids, double *w, double *logits)
{
    oracle_route_grouped(x, Wg, bias, T, H, E, k, renorm, 1, 1, ids, w, logits);
}

/* Group-limited top-k (the FusedMoE arguments use_grouped_topk,
 * num_expert_group and topk_group of the vLLM EP FusedMoE patch, _ep_init).
 * The pages name the arguments only; the reading taken here is the plainest
 * one, DeepSeek-V2's group-limited routing: the E experts form n_group groups
 * of E / n_group consecutive ids; a group's score is the largest logit of its
 * experts; the topk_group groups with the largest scores are kept (ties to
 * the lower group index); the top-k then runs over the experts of the kept
 * groups only (same order and tie rule as above).  The softmax still runs over
 * all E experts, so the weights are the same probabilities as without groups.
 * n_group <= 1 (or topk_group >= n_group) keeps every expert.
 */
void oracle_route_grouped(const uint16_t *x, const float *Wg, const float *bias,
                          int64_t T, int H, int E, int k, int renorm, int n_group, int topk_group,
                          int32_t *ids, double *w, double *logits)
{
    if (n_group < 1) n_group = 1;
    const int gsize = E / n_group;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        double *l = (double *)malloc(sizeof(double) * (size_t)E);
        char *taken = (char *)calloc((size_t)E, 1);
        char *gkeep = (char *)calloc((size_t)n_group, 1);
        double *gs = (double *)malloc(sizeof(double) * (size_t)n_group);
        const uint16_t *xt = x + (size_t)t * (size_t)H;
        for (int e = 0; e < E; ++e) {
            const float *we = Wg + (size_t)e * (size_t)H;
            double s = 0.0;
            for (int h = 0; h < H; ++h) s += oracle_bf16_to_f64(xt[h]) * (double)we[h];
            if (bias) s += (double)bias[e];
            l[e] = s;
            if (logits) logits[(size_t)t * (size_t)E + (size_t)e] = s;
        }
        /* softmax over all experts */
        double m = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp(l[e] - m);
        /* groups: score = largest logit of the group; keep topk_group of them */
        if (n_group > 1 && topk_group < n_group) {
            for (int g = 0; g < n_group; ++g) {
                double b = l[g * gsize];
                for (int e = g * gsize + 1; e < (g + 1) * gsize; ++e) if (l[e] > b) b = l[e];
                gs[g] = b;
            }
            for (int r = 0; r < topk_group; ++r) {
                int best = -1;
                for (int g = 0; g < n_group; ++g) {
                    if (gkeep[g]) continue;
                    if (best < 0 || gs[g] > gs[best]) best = g;
                }
                gkeep[best] = 1;
            }
            for (int e = 0; e < E; ++e) if (!gkeep[e / gsize]) taken[e] = 1;  /* excluded */
        }
        /* top-k: k passes of "largest remaining logit, lowest id on ties" */
        double psum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            ids[(size_t)t * (size_t)k + (size_t)j] = best;
            double p = exp(l[best] - m) / z;
            w[(size_t)t * (size_t)k + (size_t)j] = p;
            psum += p;
        }
        if (renorm)
            for (int j = 0; j < k; ++j) w[(size_t)t * (size_t)k + (size_t)j] /= psum;
        free(l);
        free(taken);
        free(gkeep);
        free(gs);
    }
}

/* ------------------------------------------------------------------------- */
/* 2. Expert -> expert slot                                                   */
/* ------------------------------------------------------------------------- */

/* Map each (token, k) pair's expert id to an expert slot.
 *
 * TensorRT-LLM PR #4495 ("large-scale EP (part 3): refactor FusedMoe for
 * redundant expert"), Description: the router computes expert ids (model side),
 * while the fused MoE op computes on expert slots (engine side), into which the
 * module loads the weights; with no mapping an expert's slot id is its id.
 * With redundant experts an expert owns rep_count[e] = rep_offset[e+1] -
 * rep_offset[e] slots, listed at rep_slots[rep_offset[e] ...], and token t uses
 * replica (t mod rep_count[e]).
 *
 *   ids [T, k]; rep_offset [E+1] or NULL (identity); rep_slots [S]
 *   slots [T, k] out
 */
void oracle_slot_map(const int32_t *ids, int64_t T, int k,
                     const int32_t *rep_offset, const int32_t *rep_slots,
                     int32_t *slots)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            size_t p = (size_t)t * (size_t)k + (size_t)j;
            int32_t e = ids[p];
            if (!rep_offset) {
                slots[p] = e;
            } else {
                int64_t c = (int64_t)rep_offset[e + 1] - (int64_t)rep_offset[e];
                slots[p] = rep_slots[rep_offset[e] + (int32_t)(t % c)];
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* 3. Expert-parallel local-range mask and remap                              */
/* ------------------------------------------------------------------------- */

/* vLLM EP FusedMoE patch, function ep_mask_and_remap: a pair is local when its
 * id lies in [start, start + count); every routing weight is multiplied by the
 * local mask (non-local pairs contribute nothing); local ids become id - start;
 * non-local ids become id mod count (MOD mode, the function as printed: the
 * pair is still computed, with weight 0) or -1 (SKIP mode: the pair is dropped,
 * the token-level skip that the function's comments attribute to the upstream
 * ragged gather).  Here the ids are expert-slot ids.
 *
 *   slots [P] in; w_in [P] in; slots_out [P] out; w_out [P] out; mask [P] out
 */
void oracle_local_mask(const int32_t *slots, const double *w_in, int64_t P,
                       int start, int count, int mode,
                       int32_t *slots_out, double *w_out, uint8_t *mask)
{
    for (int64_t p = 0; p < P; ++p) {
        int32_t s = slots[p];
        int m = (s >= start) && (s < start + count);
        w_out[p] = w_in[p] * (double)m;
        if (mask) mask[p] = (uint8_t)m;
        if (m)
            slots_out[p] = s - start;
        else
            slots_out[p] = (mode == ORACLE_NONLOCAL_MOD) ? (s % count) : -1;
    }
}

/* ------------------------------------------------------------------------- */
/* 4. Counts, offsets, permutation                                            */
/* ------------------------------------------------------------------------- */

/* Group the kept pairs by slot: counts[s] = number of pairs with slot s,
 * offsets = exclusive scan of counts (offsets[S] = total), and within a slot
 * the pairs keep ascending pair index p = t*k + j (a stable sort by slot).
 * perm_src[r] = pair placed in row r (r < offsets[S]); pair_row[p] = its row,
 * or -1 for a dropped pair (slot -1).
 *
 * The per-expert loop of the vLLM EP FusedMoE patch (module docstring: the
 * per-expert loop skips experts whose count is 0) visits exactly these groups.
 */
void oracle_permute(const int32_t *slots, int64_t P, int S,
                    int32_t *counts, int32_t *offsets,
                    int32_t *perm_src, int32_t *pair_row)
{
    for (int s = 0; s < S; ++s) counts[s] = 0;
    for (int64_t p = 0; p < P; ++p)
        if (slots[p] >= 0) counts[slots[p]] += 1;
    offsets[0] = 0;
    for (int s = 0; s < S; ++s) offsets[s + 1] = offsets[s] + counts[s];
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    for (int s = 0; s < S; ++s) next[s] = offsets[s];
    for (int64_t p = 0; p < P; ++p) {
        int32_t s = slots[p];
        if (s < 0) {
            pair_row[p] = -1;
        } else {
            int32_t r = next[s]++;
            perm_src[r] = (int32_t)p;
            pair_row[p] = r;
        }
    }
    free(next);
}

/* ------------------------------------------------------------------------- */
/* E4M3 activations                                                           */
/* ------------------------------------------------------------------------- */

/* E4M3 activations as well as weights ("W8A8"; TensorRT-LLM AutoDeploy MoE PR
 * #10985, review of torch_moe.py, names FP8 paths of the MoE ops and fixes no
 * format).  Reading: each expert input row and each intermediate row h is
 * quantised on its own, with a power-of-two scale 2^e, e the smallest integer
 * >= -126 such that amax <= 448 * 2^e (so amax / scale lies in (224, 448]
 * unless the clamp applies), and q = e4m3(v / 2^e) to nearest with ties to
 * even (the division by a power of two is exact).  An all-zero row gets
 * e = -126 and q = 0. */
void oracle_quantize_act_row(const uint16_t *v, int K, uint8_t *q, float *scale)
{
    double amax = 0.0;
    for (int c = 0; c < K; ++c) {
        const double a = fabs(oracle_bf16_to_f64(v[c]));
        if (a > amax) amax = a;
    }
    int e = -126;
    while (amax > ldexp(448.0, e)) ++e;
    *scale = (float)ldexp(1.0, e);
    for (int c = 0; c < K; ++c) q[c] = oracle_f64_to_e4m3(ldexp(oracle_bf16_to_f64(v[c]), -e));
}

void oracle_quantize_act_rows(const uint16_t *v, int64_t rows, int K, uint8_t *q, float *scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        oracle_quantize_act_row(v + (size_t)r * (size_t)K, K, q + (size_t)r * (size_t)K, scale + r);
}

/* The row v [K] as fp64 values: bf16 as is (act 0), its E4M3 quantisation
 * dequantised exactly, scale * e4m3(q) (act 1), or its NVFP4 quantisation
 * dequantised exactly, s * sb * e2m1(q), with a power-of-two s (act 2). */
static void act_values(const uint16_t *v, int K, int act, double *out)
{
    if (act == 0) {
        for (int c = 0; c < K; ++c) out[c] = oracle_bf16_to_f64(v[c]);
        return;
    }
    uint8_t *q = (uint8_t *)malloc((size_t)K);
    float sc;
    if (act == 1) {
        oracle_quantize_act_row(v, K, q, &sc);
        for (int c = 0; c < K; ++c) out[c] = (double)sc * oracle_e4m3_to_f64(q[c]);
    } else {
        uint8_t *sb = (uint8_t *)malloc((size_t)(K / 16));
        oracle_quantize_nvfp4_row(v, K, 1, q, sb, &sc);
        for (int c = 0; c < K; ++c)
            out[c] = (double)sc * oracle_e4m3_to_f64(sb[c / 16]) * oracle_e2m1_to_f64(q[c]);
        free(sb);
    }
    free(q);
}

/* ------------------------------------------------------------------------- */
/* 5. Gated MLP (SwiGLU) of one expert on one token                          */
/* ------------------------------------------------------------------------- */

/* y = W2 . bf16( silu(W1_gate . x) * (W1_up . x) ),  silu(z) = z / (1 + e^-z).
 *
 * Per-expert gated MLP as in the TensorRT-LLM AutoDeploy MoE ops (PR #10985,
 * "MoE all-to-all paradigm": is_gated_mlp / act_fn per expert) and the
 * per-expert compute of the vLLM EP FusedMoE patch.  W1 packs the gate rows
 * first and the up rows second.
 *
 *   x [H] bf16;  W1 [2I, H] bf16 (rows 0..I-1 gate, I..2I-1 up);  W2 [H, I] bf16
 *   y [H] double out;  h [I] bf16 bits out (or NULL)
 * act8: the input row and the bf16 row h are quantised to E4M3 with a
 * power-of-two scale each (oracle_quantize_act_row) before FC1 and FC2; act8 =
 * 2: to NVFP4 with a power-of-two row scale (oracle_quantize_nvfp4_row, pow2)
 * instead.
 */
static void expert_mlp_w(const uint16_t *x, const oracle_wmat *W1, const oracle_wmat *W2,
                         int H, int I, int act8, double *y, uint16_t *h_out)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)H);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)I);
    act_values(x, H, act8, xd);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int hh = 0; hh < H; ++hh) g += wget(W1, (size_t)i, (size_t)hh) * xd[hh];
        for (int hh = 0; hh < H; ++hh) u += wget(W1, (size_t)I + (size_t)i, (size_t)hh) * xd[hh];
        double a = g / (1.0 + exp(-g)) * u;
        hb[i] = oracle_f64_to_bf16(a);
        if (h_out) h_out[i] = hb[i];
    }
    act_values(hb, I, act8, h);
    for (int o = 0; o < H; ++o) {
        double s = 0.0;
        for (int i = 0; i < I; ++i) s += wget(W2, (size_t)o, (size_t)i) * h[i];
        y[o] = s;
    }
    free(xd);
    free(h);
    free(hb);
}

void oracle_expert_mlp(const uint16_t *x, const uint16_t *W1, const uint16_t *W2,
                       int H, int I, double *y, uint16_t *h_out)
{
    const oracle_wmat w1 = {W1, NULL, NULL, (size_t)H, NULL}, w2 = {W2, NULL, NULL, (size_t)I, NULL};
    expert_mlp_w(x, &w1, &w2, H, I, 0, y, h_out);
}

/* The same MLP with E4M3 weights: W1q [2I, H] with scales s1 [2I], W2q [H, I]
 * with scales s2 [H] (the dequantised values, exactly, in fp64). */
void oracle_expert_mlp_fp8(const uint16_t *x, const uint8_t *W1q, const float *s1, const uint8_t *W2q,
                           const float *s2, int H, int I, double *y, uint16_t *h_out)
{
    const oracle_wmat w1 = {NULL, W1q, s1, (size_t)H, NULL}, w2 = {NULL, W2q, s2, (size_t)I, NULL};
    expert_mlp_w(x, &w1, &w2, H, I, 0, y, h_out);
}

/* E4M3 weights and E4M3 activations (x and h quantised per row). */
void oracle_expert_mlp_w8a8(const uint16_t *x, const uint8_t *W1q, const float *s1, const uint8_t *W2q,
                            const float *s2, int H, int I, double *y, uint16_t *h_out)
{
    const oracle_wmat w1 = {NULL, W1q, s1, (size_t)H, NULL}, w2 = {NULL, W2q, s2, (size_t)I, NULL};
    expert_mlp_w(x, &w1, &w2, H, I, 1, y, h_out);
}

/* NVFP4 weights: W1q [2I, H] codes with block scales W1sb [2I, H/16] and row
 * scales s1 [2I], W2q [H, I] with W2sb [H, I/16] and s2 [H] (the dequantised
 * values, exactly, in fp64); act4: x and h quantised to NVFP4 per row too. */
void oracle_expert_mlp_nvfp4(const uint16_t *x, const uint8_t *W1q, const uint8_t *W1sb, const float *s1,
                             const uint8_t *W2q, const uint8_t *W2sb, const float *s2, int H, int I, int act4,
                             double *y, uint16_t *h_out)
{
    const oracle_wmat w1 = {NULL, W1q, s1, (size_t)H, W1sb}, w2 = {NULL, W2q, s2, (size_t)I, W2sb};
    expert_mlp_w(x, &w1, &w2, H, I, act4 ? 2 : 0, y, h_out);
}

/* ------------------------------------------------------------------------- */
/* The layer, for a list of tokens                                            */
/* ------------------------------------------------------------------------- */

/* Output rows of the MoE layer for the tokens listed in tok[0..n) (indices
 * into x; a token's result does not depend on the other tokens).
 *
 * out[t] = sum over j in 0..k-1, in order, of w_j * y_j    (kept pairs only)
 *        + g_t * sum over shared experts of y_shared
 * where w_j is the routing weight after the local mask, y_j the gated MLP of
 * the pair's slot (W1/W2 are indexed by local slot), and g_t = sigmoid(x_t .
 * w_s) when shared_gate_w is given, else 1.
 *
 * The weighted sum of the selected experts' outputs per token is the one the
 * DeepSpeed AutoTP MoE PR (#6964) reduces once per layer; the shared expert is
 * added to the routed output as in ep_reduce_output of the vLLM EP FusedMoE
 * patch (out = routed_out + shared_out).
 *
 * Weights: bf16 (W1, W2, W1s, W2s), or, where W1q / W1sq is given, E4M3 bytes
 * with one fp32 scale per row (W1q [S_local, 2I, H] + s1 [S_local, 2I], W2q
 * [S_local, H, I] + s2 [S_local, H]; the shared ones alike).  act8 (E4M3
 * weights only): the expert input rows and intermediate rows are quantised to
 * E4M3 as well (oracle_quantize_act_row), the shared experts' too.  Where the
 * block scales W1sb [S_local, 2I, H/16] / W2sb [S_local, H, I/16] (W1ssb /
 * W2ssb for the shared experts) are given, W1q ... hold NVFP4 codes instead
 * (oracle_expert_mlp_nvfp4), and act8 quantises the activations to NVFP4.
 *
 * Shared experts: n_shared experts of intermediate size I_sh each; W1s holds
 * them one after another, each [2*I_sh, H] (gate rows, then up rows); W2s holds
 * them one after another, each [H, I_sh].
 *
 * Also writes per listed token its ids / weights / slots (arrays [n, k]).
 */
void oracle_moe_tokens(const uint16_t *x, int64_t T, int H,
                       const float *Wg, const float *bias, int E, int k, int renorm,
                       int n_group, int topk_group, int on_input,
                       const int32_t *rep_offset, const int32_t *rep_slots,
                       int local_start, int local_count, int mode,
                       const uint16_t *W1, const uint16_t *W2, int I,
                       int n_shared, const uint16_t *W1s, const uint16_t *W2s, int I_sh,
                       const uint16_t *shared_gate_w,
                       const uint8_t *W1q, const float *s1, const uint8_t *W2q, const float *s2,
                       const uint8_t *W1sq, const float *s1s, const uint8_t *W2sq, const float *s2s,
                       const uint8_t *W1sb, const uint8_t *W2sb, const uint8_t *W1ssb, const uint8_t *W2ssb,
                       int act8, const int64_t *tok, int64_t n,
                       double *out, int32_t *ids_out, double *w_out, int32_t *slot_out)
{
    (void)T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < n; ++q) {
        int64_t t = tok[q];
        const uint16_t *xt = x + (size_t)t * (size_t)H;
        int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
        double *w = (double *)malloc(sizeof(double) * (size_t)k);
        int32_t *sl = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
        int32_t *sl2 = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
        double *w2 = (double *)malloc(sizeof(double) * (size_t)k);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
        double *o = out + (size_t)q * (size_t)H;

        /* steps 1-3 for this one token (the slot map needs its index t) */
        oracle_route_grouped(xt, Wg, bias, 1, H, E, k, renorm, n_group, topk_group, ids, w, NULL);
        for (int j = 0; j < k; ++j) {
            int32_t e = ids[j];
            if (!rep_offset) {
                sl[j] = e;
            } else {
                int64_t c = (int64_t)rep_offset[e + 1] - (int64_t)rep_offset[e];
                sl[j] = rep_slots[rep_offset[e] + (int32_t)(t % c)];
            }
        }
        if (local_count >= 0) {
            oracle_local_mask(sl, w, k, local_start, local_count, mode, sl2, w2, NULL);
        } else {
            for (int j = 0; j < k; ++j) { sl2[j] = sl[j]; w2[j] = w[j]; }
        }
        for (int j = 0; j < k; ++j) {
            ids_out[(size_t)q * (size_t)k + (size_t)j] = ids[j];
            w_out[(size_t)q * (size_t)k + (size_t)j] = w2[j];
            slot_out[(size_t)q * (size_t)k + (size_t)j] = sl2[j];
        }

        /* step 5: weighted sum over the k experts, in order.  With on_input the
         * routing weight scales the expert's input instead (TensorRT-LLM
         * AutoDeploy MoE PR #10985, review of torch_moe.py: apply_routing_on_input,
         * "BMM-style routing"): the row w_j * x_t, rounded to bf16, goes through
         * the expert and the outputs are summed unweighted. */
        for (int hh = 0; hh < H; ++hh) o[hh] = 0.0;
        uint16_t *xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)H);
        for (int j = 0; j < k; ++j) {
            int32_t s = sl2[j];
            if (s < 0) continue;
            const uint16_t *xin = xt;
            if (on_input) {
                for (int hh = 0; hh < H; ++hh) xs[hh] = oracle_f64_to_bf16(w2[j] * oracle_bf16_to_f64(xt[hh]));
                xin = xs;
            }
            if (W1q && W1sb)
                oracle_expert_mlp_nvfp4(xin, W1q + (size_t)s * 2u * (size_t)I * (size_t)H,
                                        W1sb + (size_t)s * 2u * (size_t)I * (size_t)(H / 16), s1 + (size_t)s * 2u * (size_t)I,
                                        W2q + (size_t)s * (size_t)H * (size_t)I,
                                        W2sb + (size_t)s * (size_t)H * (size_t)(I / 16), s2 + (size_t)s * (size_t)H,
                                        H, I, act8, y, NULL);
            else if (W1q)
                (act8 ? oracle_expert_mlp_w8a8 : oracle_expert_mlp_fp8)(xin, W1q + (size_t)s * 2u * (size_t)I * (size_t)H, s1 + (size_t)s * 2u * (size_t)I,
                                      W2q + (size_t)s * (size_t)H * (size_t)I, s2 + (size_t)s * (size_t)H, H, I, y,
                                      NULL);
            else
                oracle_expert_mlp(xin, W1 + (size_t)s * 2u * (size_t)I * (size_t)H,
                                  W2 + (size_t)s * (size_t)H * (size_t)I, H, I, y, NULL);
            const double wj = on_input ? 1.0 : w2[j];
            for (int hh = 0; hh < H; ++hh) o[hh] += wj * y[hh];
        }
        free(xs);
        if (n_shared > 0) {
            double g = 1.0;
            if (shared_gate_w) {
                double z = 0.0;
                for (int hh = 0; hh < H; ++hh)
                    z += oracle_bf16_to_f64(xt[hh]) * oracle_bf16_to_f64(shared_gate_w[hh]);
                g = 1.0 / (1.0 + exp(-z));
            }
            double *ysum = (double *)calloc((size_t)H, sizeof(double));
            for (int sidx = 0; sidx < n_shared; ++sidx) {
                if (W1sq && W1ssb)
                    oracle_expert_mlp_nvfp4(xt, W1sq + (size_t)sidx * 2u * (size_t)I_sh * (size_t)H,
                                            W1ssb + (size_t)sidx * 2u * (size_t)I_sh * (size_t)(H / 16),
                                            s1s + (size_t)sidx * 2u * (size_t)I_sh,
                                            W2sq + (size_t)sidx * (size_t)H * (size_t)I_sh,
                                            W2ssb + (size_t)sidx * (size_t)H * (size_t)(I_sh / 16),
                                            s2s + (size_t)sidx * (size_t)H, H, I_sh, act8, y, NULL);
                else if (W1sq)
                    (act8 ? oracle_expert_mlp_w8a8 : oracle_expert_mlp_fp8)(xt, W1sq + (size_t)sidx * 2u * (size_t)I_sh * (size_t)H,
                                          s1s + (size_t)sidx * 2u * (size_t)I_sh,
                                          W2sq + (size_t)sidx * (size_t)H * (size_t)I_sh, s2s + (size_t)sidx * (size_t)H,
                                          H, I_sh, y, NULL);
                else
                    oracle_expert_mlp(xt, W1s + (size_t)sidx * 2u * (size_t)I_sh * (size_t)H,
                                      W2s + (size_t)sidx * (size_t)H * (size_t)I_sh, H, I_sh, y, NULL);
                for (int hh = 0; hh < H; ++hh) ysum[hh] += y[hh];
            }
            for (int hh = 0; hh < H; ++hh) o[hh] += g * ysum[hh];
            free(ysum);
        }
        free(ids); free(w); free(sl); free(sl2); free(w2); free(y);
    }
}

/* Thread count used by the OpenMP loops above (token-parallel only; the
 * arithmetic of each token is sequential, so results do not depend on it). */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
