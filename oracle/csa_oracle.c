/*
 * CPU oracle for the CSA fused Compressor: a gated-softmax pooling over
 * THD-packed token windows, forward and backward.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
 * baseline load this file.  It shares no code, header or constant table with the
 * CUDA library; the two only meet on the inputs of csa_workloads.py.
 *
 * What it computes follows the "CSA Fused Compressor" page of the cuDNN frontend
 * documentation:
 *   - Semantics: the overlapping window form (coff == 2, window 2*ratio: positions
 *     k < ratio read the previous block's token on the first-half column j with APE
 *     row k, and are invalid for a segment's first block; positions k >= ratio read
 *     the own block's token on the second-half column head_dim + j with APE row
 *     k - ratio), the own-block form (coff == 1, window ratio, always valid), the
 *     pooling out[b, j] = sum_k kv * softmax_k(score + ape), per-segment tail
 *     tokens dropped, and rows past cu_seqlens_comp[-1] up to the static capacity
 *     computed as a segment's first block starting at token 0, with their incoming
 *     gradients ignored by the backward.
 *   - Numerics: fp32 arithmetic with one final bf16 rounding, no FMA contraction.
 *   - Class API: grad_kv / grad_score get exact zeros at every never-consumed
 *     position (segment tails, the last block's first-half columns, segments
 *     shorter than ratio, tokens outside the segments).
 *
 * Two arithmetic variants, the same loops:
 *   csa_oracle_*_f32  fp32, in one stated order (below); bf16 outputs.
 *   csa_oracle_*_f64  fp64 with libm exp(), no intermediate rounding; fp64 outputs.
 *
 * The fp32 order, per output row r and column j (the softmax written out plainly,
 * window positions in ascending k, invalid positions skipped):
 *     s_k  = f32(score) + ape                          (one rounding)
 *     m    = max_k s_k                                 (NaN if any s_k is NaN)
 *     e_k  = csa_exp_f32(s_k - m)
 *     den  = ((0 + e_0) + e_1) + ...                   (k ascending)
 *     num  = fma(e_k, f32(kv), num)                    (k ascending, from +0)
 *     inv  = 1 / den ;  o = num * inv ;  out = bf16(o)
 *   backward, real rows only, with g = f32(grad_out[r, j]):
 *     go = g * o ;  p_k = e_k * inv
 *     grad_kv    = bf16(g * p_k)
 *     ds_k       = p_k * (g * f32(kv) - go) ;  grad_score = bf16(ds_k)
 *     grad_ape[k % ratio][c] = sum over real rows, ascending, of ds_k  (fp32)
 *
 * csa_exp_f32 is this file's own exp: Cody-Waite range reduction (W. J. Cody and
 * W. Waite, "Software Manual for the Elementary Functions", 1980) with a two-part
 * ln 2, then a degree-6 polynomial of e^r on |r| <= h = ln2/2 in Horner form, then
 * scaling by 2^n through the exponent field.  Results below 2^-126.5 are +0.  The
 * polynomial is the degree-7 Taylor polynomial with its r^7 term economized over
 * |r| <= h (C. Lanczos, "Applied Analysis", 1956): with x = r/h, the Chebyshev
 * polynomial T7(x) = 64x^7 - 112x^5 + 56x^3 - 7x gives
 *     r^7 = h^7 x^7 = h^7 (T7(x) + 112x^5 - 56x^3 + 7x) / 64,
 * and dropping the T7 term (|T7| <= 1 on the interval) moves the r^7 coefficient
 * 1/7! onto r^5, r^3 and r:
 *     c5 = 1/5! + (1/7!) (112/64) h^2,   c3 = 1/3! - (1/7!) (56/64) h^4,
 *     c1 = 1 + (1/7!) (7/64) h^6  (= 1 in fp32: the change is below half an ulp),
 * the other coefficients 1/k!.  Its error, h^7/(64 7!) + the Taylor remainder
 * h^8/8!, is about 7e-9 relative (0.12 ulp), as small as the degree-7 Taylor
 * polynomial's, with one multiply-add fewer.  The coefficients are computed in
 * double from this definition and rounded to fp32.
 *
 * Build with -ffp-contract=off so that the compiler does not fuse a*b+c.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 */

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round to nearest, ties to even; NaN stays NaN; overflow goes to infinity. */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return 0x7fc0;
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ----------------------------------------------------------------- exp */

/* Constants, from their definitions:
 *   LOG2E  = 1/ln 2 rounded to fp32;
 *   LN2_HI = ln 2 with the fp32 significand cut to 16 bits (0x3F317200), so that
 *            n * LN2_HI is exact for |n| < 256;
 *   LN2_LO = ln 2 - LN2_HI rounded to fp32;
 *   MAGIC  = 1.5 * 2^23: adding it rounds a value of magnitude < 2^22 to an
 *            integer held in the low significand bits;
 *   the polynomial's coefficients (above), each rounded to fp32. */
#define CSA_LOG2E 1.44269504088896340736f
#define CSA_LN2_HI 0.693145751953125f
#define CSA_LN2_LO 1.42860682030941723212e-6f
#define CSA_MAGIC 12582912.0f
#define CSA_EXP_XMIN (-88.0f)

/* h = ln2/2 and its powers, in double */
#define CSA_H (0.69314718055994530942 / 2.0)
#define CSA_H2 (CSA_H * CSA_H)
#define CSA_H4 (CSA_H2 * CSA_H2)

float csa_oracle_exp_f32(float x)
{
    static const float c[7] = {1.0f,
                               1.0f,
                               (float)(1.0 / 2.0),
                               (float)(1.0 / 6.0 - (1.0 / 5040.0) * (56.0 / 64.0) * CSA_H4),
                               (float)(1.0 / 24.0),
                               (float)(1.0 / 120.0 + (1.0 / 5040.0) * (112.0 / 64.0) * CSA_H2),
                               (float)(1.0 / 720.0)};
    /* Clamp from below; a NaN fails the comparison and passes through. */
    float xc = (x < CSA_EXP_XMIN) ? CSA_EXP_XMIN : x;
    float t = fmaf(xc, CSA_LOG2E, CSA_MAGIC); /* MAGIC + n, n = nearest(x/ln2) */
    float nf = t - CSA_MAGIC;                 /* n as a float, exact */
    float r = fmaf(nf, -CSA_LN2_HI, xc);      /* x - n ln2, two parts */
    r = fmaf(nf, -CSA_LN2_LO, r);
    float p = c[6];
    for (int k = 5; k >= 0; --k)
        p = fmaf(p, r, c[k]);
    /* 2^n: the low bits of t hold MAGIC + n; shifting them into the exponent field
     * and adding the bias gives the bits of 2^n (n = -127 gives +0). */
    uint32_t tb;
    memcpy(&tb, &t, 4);
    uint32_t sb = tb * 8388608u + 0x3f800000u;
    float scale;
    memcpy(&scale, &sb, 4);
    return p * scale;
}

/* ------------------------------------------------------------- windows */

typedef struct {
    int real;      /* row r < cu_seqlens_comp[n_seg] */
    int64_t base;  /* first token of the row's own block */
    int first;     /* first block of its segment (or a padding row) */
} row_info;

/* Row r belongs to segment s with cu_seqlens_comp[s] <= r < cu_seqlens_comp[s+1]; it
 * is that segment's block b = r - cu_seqlens_comp[s], whose own tokens start at
 * cu_seqlens[s] + b*ratio.  Rows at or past cu_seqlens_comp[n_seg] are padding
 * rows: a first block whose own tokens start at token 0. */
static row_info row_of(int64_t r, const int32_t *cu_seqlens, const int32_t *cu_comp,
                       int32_t n_seg, int32_t ratio)
{
    row_info ri = {0, 0, 1};
    for (int32_t s = 0; s < n_seg; ++s) {
        if (cu_comp[s] <= r && r < cu_comp[s + 1]) {
            int64_t b = r - cu_comp[s];
            ri.real = 1;
            ri.base = (int64_t)cu_seqlens[s] + b * ratio;
            ri.first = (b == 0);
            return ri;
        }
    }
    return ri;
}

typedef struct {
    int valid;
    int64_t token;
    int64_t col;     /* packed column in [0, coff*head_dim) */
    int64_t ape_row; /* k % ratio */
} slot;

/* Window position k of a row, for output column j (Semantics section). */
static slot slot_of(const row_info *ri, int32_t k, int64_t j, int32_t ratio, int32_t coff,
                    int32_t head_dim)
{
    slot sl;
    if (coff == 2 && k < ratio) {
        /* previous block's token, first-half column, APE row k */
        sl.valid = !ri->first;
        sl.token = ri->base - ratio + k;
        sl.col = j;
        sl.ape_row = k;
    } else if (coff == 2) {
        /* own block's token, second-half column, APE row k - ratio */
        sl.valid = 1;
        sl.token = ri->base + (k - ratio);
        sl.col = head_dim + j;
        sl.ape_row = k - ratio;
    } else {
        /* own-block form: own token, column j, APE row k */
        sl.valid = 1;
        sl.token = ri->base + k;
        sl.col = j;
        sl.ape_row = k;
    }
    return sl;
}

static int check_args(int32_t n_seg, int32_t ratio, int32_t coff, int32_t head_dim,
                      int32_t capacity)
{
    if (n_seg < 0 || ratio < 1 || (coff != 1 && coff != 2) || head_dim < 1 || capacity < 0)
        return -1;
    return 0;
}

/* ------------------------------------------------------ fp32, one order */

/* One (row, column) of the fp32 forward.  Fills e[k] (0 at invalid k), returns o
 * (the fp32 output before its bf16 rounding) and inv = 1/den. */
static float pool_f32(const uint16_t *kv, const uint16_t *score, const float *ape,
                      const row_info *ri, int64_t j, int32_t ratio, int32_t coff,
                      int32_t head_dim, float *e, float *inv_out)
{
    const int32_t W = coff * ratio;
    const int64_t C = (int64_t)coff * head_dim;
    float m = -INFINITY;
    int saw_nan = 0;
    for (int32_t k = 0; k < W; ++k) {
        slot sl = slot_of(ri, k, j, ratio, coff, head_dim);
        if (!sl.valid)
            continue;
        float s = bf16_to_f32(score[sl.token * C + sl.col]) + ape[sl.ape_row * C + sl.col];
        e[k] = s; /* holds s_k until the second pass */
        if (isnan(s))
            saw_nan = 1;
        else if (s > m)
            m = s;
    }
    if (saw_nan)
        m = NAN;
    float den = 0.0f, num = 0.0f;
    for (int32_t k = 0; k < W; ++k) {
        slot sl = slot_of(ri, k, j, ratio, coff, head_dim);
        if (!sl.valid) {
            e[k] = 0.0f;
            continue;
        }
        float ek = csa_oracle_exp_f32(e[k] - m);
        e[k] = ek;
        den = den + ek;
        num = fmaf(ek, bf16_to_f32(kv[sl.token * C + sl.col]), num);
    }
    float inv = 1.0f / den;
    *inv_out = inv;
    return num * inv;
}

int csa_oracle_fwd_f32(const uint16_t *kv, const uint16_t *score, const float *ape,
                       const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp,
                       int32_t n_seg, int32_t ratio, int32_t coff, int32_t head_dim,
                       int32_t capacity, uint16_t *out)
{
    if (check_args(n_seg, ratio, coff, head_dim, capacity))
        return -1;
    float *e = (float *)malloc(sizeof(float) * (size_t)(coff * ratio));
    if (!e)
        return -2;
    for (int64_t r = 0; r < capacity; ++r) {
        row_info ri = row_of(r, cu_seqlens, cu_seqlens_comp, n_seg, ratio);
        for (int64_t j = 0; j < head_dim; ++j) {
            float inv;
            float o = pool_f32(kv, score, ape, &ri, j, ratio, coff, head_dim, e, &inv);
            out[r * head_dim + j] = f32_to_bf16(o);
        }
    }
    free(e);
    return 0;
}

/* Backward.  n_tokens rows of grad_kv / grad_score are written: zeros everywhere,
 * then the consumed slots.  Padding rows contribute nothing. */
int csa_oracle_bwd_f32(const uint16_t *kv, const uint16_t *score, const float *ape,
                       const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp,
                       int32_t n_seg, int32_t ratio, int32_t coff, int32_t head_dim,
                       int32_t capacity, int64_t n_tokens, const uint16_t *grad_out,
                       uint16_t *dkv, uint16_t *dscore, float *dape)
{
    if (check_args(n_seg, ratio, coff, head_dim, capacity) || n_tokens < 0)
        return -1;
    const int32_t W = coff * ratio;
    const int64_t C = (int64_t)coff * head_dim;
    memset(dkv, 0, sizeof(uint16_t) * (size_t)(n_tokens * C));
    memset(dscore, 0, sizeof(uint16_t) * (size_t)(n_tokens * C));
    for (int64_t i = 0; i < (int64_t)ratio * C; ++i)
        dape[i] = 0.0f;
    float *e = (float *)malloc(sizeof(float) * (size_t)W);
    if (!e)
        return -2;
    for (int64_t r = 0; r < capacity; ++r) {
        row_info ri = row_of(r, cu_seqlens, cu_seqlens_comp, n_seg, ratio);
        if (!ri.real)
            continue; /* padding rows: incoming gradient ignored */
        for (int64_t j = 0; j < head_dim; ++j) {
            float inv;
            float o = pool_f32(kv, score, ape, &ri, j, ratio, coff, head_dim, e, &inv);
            float g = bf16_to_f32(grad_out[r * head_dim + j]);
            float go = g * o;
            for (int32_t k = 0; k < W; ++k) {
                slot sl = slot_of(&ri, k, j, ratio, coff, head_dim);
                if (!sl.valid)
                    continue;
                float p = e[k] * inv;
                float v = bf16_to_f32(kv[sl.token * C + sl.col]);
                float ds = p * (g * v - go);
                dkv[sl.token * C + sl.col] = f32_to_bf16(g * p);
                dscore[sl.token * C + sl.col] = f32_to_bf16(ds);
                dape[sl.ape_row * C + sl.col] += ds;
            }
        }
    }
    free(e);
    return 0;
}

/* ------------------------------------------------------------- fp64 */

static double pool_f64(const uint16_t *kv, const uint16_t *score, const float *ape,
                       const row_info *ri, int64_t j, int32_t ratio, int32_t coff,
                       int32_t head_dim, double *p)
{
    const int32_t W = coff * ratio;
    const int64_t C = (int64_t)coff * head_dim;
    double m = -INFINITY;
    int saw_nan = 0;
    for (int32_t k = 0; k < W; ++k) {
        slot sl = slot_of(ri, k, j, ratio, coff, head_dim);
        if (!sl.valid)
            continue;
        double s = (double)bf16_to_f32(score[sl.token * C + sl.col]) +
                   (double)ape[sl.ape_row * C + sl.col];
        p[k] = s;
        if (isnan(s))
            saw_nan = 1;
        else if (s > m)
            m = s;
    }
    if (saw_nan)
        m = NAN;
    double den = 0.0;
    for (int32_t k = 0; k < W; ++k) {
        slot sl = slot_of(ri, k, j, ratio, coff, head_dim);
        if (!sl.valid) {
            p[k] = 0.0;
            continue;
        }
        p[k] = exp(p[k] - m);
        den += p[k];
    }
    double o = 0.0;
    for (int32_t k = 0; k < W; ++k) {
        slot sl = slot_of(ri, k, j, ratio, coff, head_dim);
        if (!sl.valid)
            continue;
        p[k] = p[k] / den;
        o += p[k] * (double)bf16_to_f32(kv[sl.token * C + sl.col]);
    }
    return o;
}

int csa_oracle_fwd_f64(const uint16_t *kv, const uint16_t *score, const float *ape,
                       const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp,
                       int32_t n_seg, int32_t ratio, int32_t coff, int32_t head_dim,
                       int32_t capacity, double *out)
{
    if (check_args(n_seg, ratio, coff, head_dim, capacity))
        return -1;
    double *p = (double *)malloc(sizeof(double) * (size_t)(coff * ratio));
    if (!p)
        return -2;
    for (int64_t r = 0; r < capacity; ++r) {
        row_info ri = row_of(r, cu_seqlens, cu_seqlens_comp, n_seg, ratio);
        for (int64_t j = 0; j < head_dim; ++j)
            out[r * head_dim + j] = pool_f64(kv, score, ape, &ri, j, ratio, coff, head_dim, p);
    }
    free(p);
    return 0;
}

/* fp64 backward of the fp64 forward.  dape_abs (may be NULL) receives, per APE
 * entry, the sum of |ds| over its contributions: the scale of the entry's
 * summation error bound. */
int csa_oracle_bwd_f64(const uint16_t *kv, const uint16_t *score, const float *ape,
                       const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp,
                       int32_t n_seg, int32_t ratio, int32_t coff, int32_t head_dim,
                       int32_t capacity, int64_t n_tokens, const uint16_t *grad_out,
                       double *dkv, double *dscore, double *dape, double *dape_abs)
{
    if (check_args(n_seg, ratio, coff, head_dim, capacity) || n_tokens < 0)
        return -1;
    const int32_t W = coff * ratio;
    const int64_t C = (int64_t)coff * head_dim;
    for (int64_t i = 0; i < n_tokens * C; ++i) {
        dkv[i] = 0.0;
        dscore[i] = 0.0;
    }
    for (int64_t i = 0; i < (int64_t)ratio * C; ++i) {
        dape[i] = 0.0;
        if (dape_abs)
            dape_abs[i] = 0.0;
    }
    double *p = (double *)malloc(sizeof(double) * (size_t)W);
    if (!p)
        return -2;
    for (int64_t r = 0; r < capacity; ++r) {
        row_info ri = row_of(r, cu_seqlens, cu_seqlens_comp, n_seg, ratio);
        if (!ri.real)
            continue;
        for (int64_t j = 0; j < head_dim; ++j) {
            double o = pool_f64(kv, score, ape, &ri, j, ratio, coff, head_dim, p);
            double g = (double)bf16_to_f32(grad_out[r * head_dim + j]);
            for (int32_t k = 0; k < W; ++k) {
                slot sl = slot_of(&ri, k, j, ratio, coff, head_dim);
                if (!sl.valid)
                    continue;
                double v = (double)bf16_to_f32(kv[sl.token * C + sl.col]);
                double ds = p[k] * g * (v - o);
                dkv[sl.token * C + sl.col] = g * p[k];
                dscore[sl.token * C + sl.col] = ds;
                dape[sl.ape_row * C + sl.col] += ds;
                if (dape_abs)
                    dape_abs[sl.ape_row * C + sl.col] += fabs(ds);
            }
        }
    }
    free(p);
    return 0;
}

/* ------------------------------------------------------- introspection */

/* Which row consumes each (token, packed column): -1 if none, -2 if more than one.
 * Lets the tests check that every slot is read by at most one real row. */
int csa_oracle_consumers(const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp,
                         int32_t n_seg, int32_t ratio, int32_t coff, int32_t head_dim,
                         int32_t capacity, int64_t n_tokens, int64_t *owner)
{
    if (check_args(n_seg, ratio, coff, head_dim, capacity) || n_tokens < 0)
        return -1;
    const int64_t C = (int64_t)coff * head_dim;
    for (int64_t i = 0; i < n_tokens * C; ++i)
        owner[i] = -1;
    for (int64_t r = 0; r < capacity; ++r) {
        row_info ri = row_of(r, cu_seqlens, cu_seqlens_comp, n_seg, ratio);
        if (!ri.real)
            continue;
        for (int64_t j = 0; j < head_dim; ++j)
            for (int32_t k = 0; k < coff * ratio; ++k) {
                slot sl = slot_of(&ri, k, j, ratio, coff, head_dim);
                if (!sl.valid)
                    continue;
                if (sl.token < 0 || sl.token >= n_tokens)
                    return -3;
                int64_t *o = &owner[sl.token * C + sl.col];
                *o = (*o == -1) ? r : -2;
            }
    }
    return 0;
}

/* ------------------------------------------- grad_ape in a stated grouping */

/* The pages fix grad_ape only as a sum over the real rows (Semantics: the chain
 * rule through the pooling) and ask that it be deterministic (Numerics).  How the
 * rows are grouped for that sum is the implementation's choice.  This function
 * evaluates the first level of any grouping plainly: leaf_of_row[r] names the
 * leaf (0 <= leaf < n_leaves) that real row r belongs to, and each leaf is the fp32
 * sum, from +0 in ascending row order, of the ds values of its rows -- the same ds
 * as csa_oracle_bwd_f32 computes.  leaves is [n_leaves][ratio][coff*head_dim].
 * Every real row must name a leaf (the sum takes each row exactly once); rows at
 * or past cu_seqlens_comp[n_seg] are padding rows and are not read.  How leaves
 * combine into grad_ape is left to the caller. */
int csa_oracle_dape_leaves_f32(const uint16_t *kv, const uint16_t *score, const float *ape,
                               const int32_t *cu_seqlens, const int32_t *cu_seqlens_comp,
                               int32_t n_seg, int32_t ratio, int32_t coff, int32_t head_dim,
                               int32_t capacity, const uint16_t *grad_out,
                               const int32_t *leaf_of_row, int32_t n_leaves, float *leaves)
{
    if (check_args(n_seg, ratio, coff, head_dim, capacity) || n_leaves < 1)
        return -1;
    const int32_t W = coff * ratio;
    const int64_t C = (int64_t)coff * head_dim;
    for (int64_t i = 0; i < (int64_t)n_leaves * ratio * C; ++i)
        leaves[i] = 0.0f;
    float *e = (float *)malloc(sizeof(float) * (size_t)W);
    if (!e)
        return -2;
    for (int64_t r = 0; r < capacity; ++r) {
        row_info ri = row_of(r, cu_seqlens, cu_seqlens_comp, n_seg, ratio);
        if (!ri.real)
            continue;
        const int32_t leaf = leaf_of_row[r];
        if (leaf < 0 || leaf >= n_leaves) {
            free(e);
            return -3;
        }
        float *acc = leaves + (int64_t)leaf * ratio * C;
        for (int64_t j = 0; j < head_dim; ++j) {
            float inv;
            float o = pool_f32(kv, score, ape, &ri, j, ratio, coff, head_dim, e, &inv);
            float g = bf16_to_f32(grad_out[r * head_dim + j]);
            float go = g * o;
            for (int32_t k = 0; k < W; ++k) {
                slot sl = slot_of(&ri, k, j, ratio, coff, head_dim);
                if (!sl.valid)
                    continue;
                float p = e[k] * inv;
                float v = bf16_to_f32(kv[sl.token * C + sl.col]);
                float ds_k = p * (g * v - go);
                acc[sl.ape_row * C + sl.col] += ds_k;
            }
        }
    }
    free(e);
    return 0;
}
