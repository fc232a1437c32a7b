/*
 * oracle.c -- plain, slow CPU oracle for the quantized MoE expert projection.
 *
 * TEST INFRASTRUCTURE. This file is the reference the CUDA path is checked against.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load it; the
 * library's product path never includes, links or calls anything here, and this file
 * includes nothing from the library.
 *
 * What it follows (docs.rs source pages of the memra-engine crate):
 *   [Q]  memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs, fn quant_rows
 *        (per-row, per-128 FP8-E4M3 activation quantisation, all in f32).
 *   [R]  same page, fn f64_ref (f64-ordered reference of the quantised GEMM plus the
 *        per-output sum of |scaled products| used by the error model).
 *   [D]  memra-engine 0.71.0, src/bin/kernel_check.rs, the F8-E4M3 MMVQ section's CPU
 *        e4m3 decode closure (sign / 4-bit exponent, bias 7 / 3-bit mantissa,
 *        exponent 0 -> subnormal, exponent 15 with mantissa 7 -> NaN).
 *   [S]  same page as [Q]: struct ExpertRaw (nibble pairs [n,k/2], low nibble = even k;
 *        e4m3 scale per 16 (NVFP4) or e8m0 scale per 32 (MXFP4); f32 scale2 for NVFP4).
 *   [M]  same page as [Q], fn mirror_gemm: the summation order of the page's own GPU
 *        kernel, in f32, restated as a specification where it is implemented below.
 *   [C]  memra-engine 0.71.0, src/bin/kernel_check.rs, grouped MoE GEMM section: routed
 *        rows grouped by expert behind CSR offsets, offsets[e+1] = offsets[e] + rows of e,
 *        and a per-routed-row factor applied to that row's output.
 *   [T]  memra-engine 0.125.0, src/bin/qwen4exp_gpu_gate.rs, the device-router arm: a
 *        softmax top-k router (selected ids and their order exact, weights within a few
 *        ulps). Its body is not printed; the reading taken is stated at orc_route_topk.
 *   [G]  same page as [Q], the swiglu_limit saturation cell and the f64 check of main:
 *        h = g * (1 / (1 + exp(-g))) * u with u = clamp(up, -L, L) and g = min(gate, L)
 *        (up clamped on both sides, gate on one side, both before the sigmoid).
 *   [W]  memra-engine 0.71.0, src/bin/kernel_check.rs, the NVFP4 W4A4 MMQ GEMM section:
 *        E2M1 activations with two-level scaling (a per-token row scale from the row amax,
 *        applied after the sum, and a UE4M3 micro-scale of amax_sub / 6 per 16 values), the
 *        sub-block-only quantiser ("V1") it is compared with, and the dynamic-range arm
 *        where the row scale must beat sub-block-only scaling per token.
 *
 * Readings for [W] (the page names the two levels but prints neither formula):
 *   row scale      r = amax_row / (6 * 448) in f32, so that the loudest sub-block's
 *                  micro-scale lands on the top of the e4m3 range; r = 0 for a zero row,
 *                  whose codes and micro-scales are all zero.
 *   normalised row y = x / r (f32), sub-block amax m = max |y| over its 16 values.
 *   micro-scale    s = e4m3 code nearest to m / 6 (f32 division, then the e4m3 encoding
 *                  above, ties to the even code); S its value.
 *   code           E2M1 value nearest to y / S (f32 division), ties to the even code,
 *                  magnitudes above 6 saturate to 6, sign kept (negative values that
 *                  round to zero give the code 0x8); every code of a block with S = 0 is 0.
 *   V1             the same without the row scale: s = nearest e4m3 code to amax_sub / 6,
 *                  raised to the smallest positive code (0x01) when that rounds to zero and
 *                  amax_sub > 0 (the page: the micro-scale clamps), saturating at 448.
 *   The page's "/2 in ue4m3_to_fp32" belongs to a storage that keeps the E2M1 grid doubled;
 *   with the plain E2M1 grid used here the micro-scale is the plain e4m3 value.
 *   Dequantised activation x^ = E2M1(code) * S * r; the W4A4 reference is f64 over
 *   x^ and the NVFP4 weight E2M1 * e4m3 * scale2, every product exact.
 *
 * Readings where the pages import a helper without printing it (each is a plain
 * definition written out here):
 *   pow2_ceil(x)       smallest power of two >= x (x > 0, finite).
 *   f32_to_fp8_e4m3(v) nearest finite e4m3fn value, ties to the even code, sign kept
 *                      (so -0.0 and negative values that round to zero give 0x80);
 *                      callers clamp to [-448, 448] first, as [Q] does.
 *   E2M1[c]            the OCP E2M1 element: 1 sign, 2 exponent bits (bias 1),
 *                      1 mantissa bit, exponent 0 subnormal; no inf/NaN.
 *   e8m0_to_f32(e)     2^(e-127); e = 255 is NaN.
 * All four minifloat decoders go through one generic sign/exponent/mantissa decoder.
 *
 * Precision: [Q] fixes f32 arithmetic (amax, amax*inv, v/s, clamp) and it is kept in
 * f32 here; [R] is f64 with the per-group weight scale first rounded in f32, kept too.
 * [G] is evaluated in f64 (the page's f32 evaluation differs from it by a few ulps, the
 * class its GPU check allows).
 * Build with -O2 -ffp-contract=off (no fused multiply-add contraction).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

/* ------------------------------------------------------------------ minifloats */

/* Decode `bits` as a sign / ebits exponent / mbits mantissa minifloat with the given
 * bias; exponent field 0 is subnormal. No special values here (callers add them). */
static double minifloat_decode(unsigned bits, int ebits, int mbits, int bias)
{
    const unsigned sign = (bits >> (ebits + mbits)) & 1u;
    const unsigned e = (bits >> mbits) & ((1u << ebits) - 1u);
    const unsigned m = bits & ((1u << mbits) - 1u);
    double mag;
    if (e == 0)
        mag = ldexp((double)m, 1 - bias - mbits);
    else
        mag = ldexp((double)((1u << mbits) | m), (int)e - bias - mbits);
    return sign ? -mag : mag;
}

double orc_e4m3_decode(uint8_t b)
{
    /* [D]: exponent 15 with mantissa 7 is NaN; no infinities (e4m3fn). */
    if ((b & 0x7Fu) == 0x7Fu)
        return NAN;
    return minifloat_decode(b, 4, 3, 7);
}

double orc_e2m1_decode(uint8_t nib)
{
    return minifloat_decode(nib & 0x0Fu, 2, 1, 1);
}

double orc_e8m0_decode(uint8_t e)
{
    if (e == 0xFFu)
        return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* Decode tables, filled once from the decoders above (speed only). */
static double g_e4m3[256];
static double g_e2m1[16];
static double g_grid[127]; /* non-negative finite e4m3 values, codes 0x00..0x7E */
static int g_init = 0;

static void init_tables(void)
{
    if (g_init)
        return;
    for (int c = 0; c < 256; ++c)
        g_e4m3[c] = orc_e4m3_decode((uint8_t)c);
    for (int c = 0; c < 16; ++c)
        g_e2m1[c] = orc_e2m1_decode((uint8_t)c);
    for (int c = 0; c < 127; ++c)
        g_grid[c] = g_e4m3[c];
    g_init = 1;
}

uint8_t orc_e4m3_encode(float v)
{
    /* Nearest value of the finite e4m3 grid, ties to the even code. Codes 0x00..0x7E
     * are strictly increasing in value, so a bisection finds the bracketing pair. */
    init_tables();
    const int neg = signbit(v) ? 1 : 0;
    const double a = fabs((double)v);
    int c;
    if (a >= g_grid[126]) {
        c = 126; /* |v| = 448 under [Q]'s clamp; the W4A4 micro-scale can pass 448 by an ulp */
    } else {
        int lo = 0, hi = 126; /* invariant: g_grid[lo] <= a < g_grid[hi] */
        while (hi - lo > 1) {
            const int mid = (lo + hi) / 2;
            if (g_grid[mid] <= a)
                lo = mid;
            else
                hi = mid;
        }
        const double dlo = a - g_grid[lo];
        const double dhi = g_grid[hi] - a;
        if (dhi < dlo || (dhi == dlo && (hi & 1) == 0))
            c = hi;
        else
            c = lo;
    }
    return (uint8_t)(c | (neg ? 0x80 : 0x00));
}

float orc_pow2_ceil(float x)
{
    /* Smallest power of two >= x, for finite x > 0: x = f * 2^e with f in [0.5, 1). */
    int e;
    const double f = frexp((double)x, &e);
    if (f == 0.5)
        return x;
    return (float)ldexp(1.0, e);
}

/* ------------------------------------------------------------------ act_quant [Q] */

void orc_act_quant(const float *x, int64_t rows, int64_t k, uint8_t *codes, float *scales)
{
    init_tables();
    const int64_t kq = k / 128;
    const float inv = (float)(1.0 / 448.0);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < kq; ++g) {
            const float *grp = x + r * k + g * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                const float a = fabsf(grp[i]);
                if (a > amax)
                    amax = a;
            }
            if (amax < 1e-4f)
                amax = 1e-4f;
            const float t = amax * inv;
            const float s = orc_pow2_ceil(t);
            scales[r * kq + g] = s;
            for (int i = 0; i < 128; ++i) {
                float q = grp[i] / s;
                if (q < -448.0f)
                    q = -448.0f;
                if (q > 448.0f)
                    q = 448.0f;
                codes[r * k + g * 128 + i] = orc_e4m3_encode(q);
            }
        }
    }
}

/* ------------------------------------------------------------------ GEMM reference [R] */

static int group_size(int recipe)
{
    return recipe == ORC_NVFP4 ? 16 : 32;
}

/* Per-group weight scale `ws` exactly as [R] forms it: NVFP4 rounds e4m3 * scale2 in f32. */
static float weight_scale(int recipe, uint8_t scbyte, float scale2)
{
    if (recipe == ORC_NVFP4)
        return (float)g_e4m3[scbyte] * scale2;
    return (float)orc_e8m0_decode(scbyte);
}

/* One output of [R]: activation row `arow` (codes) with its per-128 scales `asrow`
 * against weight column `col` of one expert. */
static void ref_one(const uint8_t *arow, const float *asrow, const uint8_t *w, const uint8_t *sc,
                    float scale2, int recipe, int64_t k, int64_t col, double *out, double *absp)
{
    const int gs = group_size(recipe);
    const int64_t ngroups = k / gs;
    const uint8_t *wrow = w + col * (k / 2);
    const uint8_t *srow = sc + col * ngroups;
    double acc = 0.0, aabs = 0.0;
    for (int64_t j = 0; j < ngroups; ++j) {
        const double ws = (double)weight_scale(recipe, srow[j], scale2);
        const double scl = ws * (double)asrow[(j * gs) / 128];
        for (int i = 0; i < gs; ++i) {
            const int64_t kk = j * gs + i;
            const uint8_t byte = wrow[kk >> 1];
            const uint8_t nib = (kk & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0x0F);
            const double p = g_e4m3[arow[kk]] * g_e2m1[nib] * scl;
            acc += p;
            aabs += fabs(p);
        }
    }
    *out = acc;
    *absp = aabs;
}

void orc_gemm_ref(const uint8_t *codes, const float *scales, const uint8_t *w, const uint8_t *sc,
                  float scale2, int recipe, int64_t g, int64_t n, int64_t k, double *out,
                  double *absp)
{
    init_tables();
    const int64_t kq = k / 128;
    for (int64_t row = 0; row < g; ++row)
        for (int64_t col = 0; col < n; ++col)
            ref_one(codes + row * k, scales + row * kq, w, sc, scale2, recipe, k, col,
                    out + row * n + col, absp + row * n + col);
}

/* ------------------------------------------------------------------ grouped, sampled */

/* Expert owning routed row p under CSR offsets (offsets[e] <= p < offsets[e+1]). */
static int expert_of(const int32_t *offsets, int num_experts, int64_t p)
{
    for (int e = 0; e < num_experts; ++e)
        if (p >= offsets[e] && p < offsets[e + 1])
            return e;
    return -1;
}

int orc_grouped_ref_sampled(const float *x, int64_t T, int64_t k, const int32_t *row_ids,
                            const int32_t *offsets, int num_experts, int64_t P, const uint8_t *w,
                            const uint8_t *sc, const float *scale2, int recipe, int64_t n,
                            const int64_t *sample_p, const int64_t *sample_col, int64_t ns,
                            double *out, double *absp, uint8_t *tmp_codes, float *tmp_scales)
{
    /* Routed row p is x[row_ids[p]] (or x[p] without row_ids), quantised by [Q] and
     * multiplied by [R] against the weights of the expert whose offset range holds p.
     * tmp_codes [k] and tmp_scales [k/128] are caller scratch. Returns 0, or -1 on a
     * row id / offset outside its range. */
    init_tables();
    const int gs = group_size(recipe);
    const int64_t wbytes = n * (k / 2);
    const int64_t sbytes = n * (k / gs);
    int64_t cur_p = -1;
    int cur_e = -1;
    for (int64_t s = 0; s < ns; ++s) {
        const int64_t p = sample_p[s];
        if (p < 0 || p >= P)
            return -1;
        if (p != cur_p) {
            const int64_t t = row_ids ? (int64_t)row_ids[p] : p;
            if (t < 0 || t >= T)
                return -1;
            cur_e = expert_of(offsets, num_experts, p);
            if (cur_e < 0)
                return -1;
            orc_act_quant(x + t * k, 1, k, tmp_codes, tmp_scales);
            cur_p = p;
        }
        const int64_t col = sample_col[s];
        if (col < 0 || col >= n)
            return -1;
        const float s2 = (recipe == ORC_NVFP4) ? scale2[cur_e] : 0.0f;
        ref_one(tmp_codes, tmp_scales, w + (int64_t)cur_e * wbytes, sc + (int64_t)cur_e * sbytes,
                s2, recipe, k, col, out + s, absp + s);
    }
    return 0;
}

/* ------------------------------------------------------------------ SwiGLU [G] */

void orc_swiglu(const float *gate, const float *up, int64_t ld, int64_t rows, int64_t inter,
                float limit, double *h)
{
    const double L = (double)limit;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < inter; ++i) {
            double u = (double)up[r * ld + i];
            if (u < -L)
                u = -L;
            if (u > L)
                u = L;
            double g = (double)gate[r * ld + i];
            if (g > L)
                g = L;
            h[r * inter + i] = g * (1.0 / (1.0 + exp(-g))) * u;
        }
    }
}

/* ------------------------------------------------------------------ mirror order [M] */

/*
 * The summation order of the page's own kernel, restated as a specification:
 *   group term  G_j = (the gs exact products e4m3(code) * E2M1(nibble) of weight group j,
 *                     added one at a time in k order, in f32) * f32(ws_j * s_a), with s_a
 *                     the scale of the activation block that holds the group;
 *   partial     P_t = the f32 running sum of G_t, G_{t+128}, G_{t+256}, ..., in that order
 *                     (starting from 0);
 *   result          = P_0 after the levels w = 64, 32, ..., 1 of a pairwise tree, each
 *                     replacing P_t by P_t + P_{t+w} for every t < w.
 * Below: all group terms of an output first, then the strided fold, then the tree.
 */
#define ORC_MIRROR_WIDTH 128

static float mirror_group_term(const uint8_t *codes_row, const float *scales_row,
                               const uint8_t *nibbles, uint8_t scale_byte, float scale2,
                               int recipe, int gs, int64_t j)
{
    float dot = 0.0f;
    for (int64_t kk = j * gs; kk < (j + 1) * gs; ++kk) {
        const unsigned nib = (unsigned)(nibbles[kk / 2] >> (4 * (kk % 2))) & 0x0Fu;
        const float a = (float)g_e4m3[codes_row[kk]];
        const float wv = (float)g_e2m1[nib];
        dot = dot + a * wv; /* the product is exact in f32; one rounding per add */
    }
    const float ws = weight_scale(recipe, scale_byte, scale2);
    return dot * (ws * scales_row[(j * gs) / 128]);
}

void orc_mirror_gemm(const uint8_t *codes, const float *scales, const uint8_t *w,
                     const uint8_t *sc, float scale2, int recipe, int64_t g, int64_t n, int64_t k,
                     float *out)
{
    init_tables();
    const int gs = group_size(recipe);
    const int64_t groups = k / gs;
    float *terms = (float *)malloc((size_t)groups * sizeof(float));
    float part[ORC_MIRROR_WIDTH];
    if (!terms)
        return;
    for (int64_t r = 0; r < g; ++r) {
        for (int64_t c = 0; c < n; ++c) {
            for (int64_t j = 0; j < groups; ++j)
                terms[j] = mirror_group_term(codes + r * k, scales + r * (k / 128),
                                             w + c * (k / 2), sc[c * groups + j], scale2, recipe,
                                             gs, j);
            for (int t = 0; t < ORC_MIRROR_WIDTH; ++t) {
                part[t] = 0.0f;
                for (int64_t j = t; j < groups; j += ORC_MIRROR_WIDTH)
                    part[t] = part[t] + terms[j];
            }
            for (int width = ORC_MIRROR_WIDTH / 2; width >= 1; width /= 2)
                for (int t = 0; t < width; ++t)
                    part[t] = part[t] + part[t + width];
            out[r * n + c] = part[0];
        }
    }
    free(terms);
}

/* ------------------------------------------------------------------ routing front-end [T] [C] */

/*
 * Router [T] (reading): each token picks the topk experts with the largest logits (a
 * softmax is monotone, so these are also the largest probabilities); equal logits rank the
 * lower expert id first; ids are emitted best first. Weights are softmax probabilities in
 * f64: p_e = exp(l_e - max) / sum_e' exp(l_e' - max) over all E experts, or, with
 * renormalize, the selected ones divided by their sum.
 */
void orc_route_topk(const float *logits, int64_t T, int E, int topk, int renormalize,
                    int32_t *ids, double *weights)
{
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        int32_t *id = ids + t * topk;
        for (int j = 0; j < topk; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                int taken = 0;
                for (int i = 0; i < j; ++i)
                    taken |= (id[i] == e);
                if (!taken && (best < 0 || l[e] > l[best]))
                    best = e; /* strictly greater: the lower id keeps a tie */
            }
            id[j] = best;
        }
        double mx = -INFINITY;
        for (int e = 0; e < E; ++e)
            if ((double)l[e] > mx)
                mx = (double)l[e];
        double denom = 0.0;
        if (renormalize) {
            for (int j = 0; j < topk; ++j)
                denom += exp((double)l[id[j]] - mx);
        } else {
            for (int e = 0; e < E; ++e)
                denom += exp((double)l[e] - mx);
        }
        for (int j = 0; j < topk; ++j)
            weights[t * topk + j] = exp((double)l[id[j]] - mx) / denom;
    }
}

/*
 * CSR construction [C]: routed rows grouped by expert, in token order within an expert (a
 * counting sort of the (token, slot) pairs by expert id, stable in token order).
 * ids [T, topk] -> offsets [E+1], row_ids [T*topk] (the token of each routed row) and
 * pair_rows [T, topk] (the routed row of each pair). Returns 0, or -1 if an id is outside
 * [0, E).
 */
int orc_route_csr(const int32_t *ids, int64_t T, int topk, int E, int32_t *offsets,
                  int32_t *row_ids, int32_t *pair_rows)
{
    for (int e = 0; e <= E; ++e)
        offsets[e] = 0;
    for (int64_t i = 0; i < T * topk; ++i) {
        if (ids[i] < 0 || ids[i] >= E)
            return -1;
        offsets[ids[i] + 1] += 1;
    }
    for (int e = 0; e < E; ++e)
        offsets[e + 1] += offsets[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!fill)
        return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < topk; ++j) {
            const int e = ids[t * topk + j];
            const int32_t p = offsets[e] + fill[e]++;
            row_ids[p] = (int32_t)t;
            pair_rows[t * topk + j] = p;
        }
    free(fill);
    return 0;
}

/*
 * Weighted combine [C]: y[t][c] = sum over the token's pairs j of weight[t][j] *
 * out[pair_rows[t][j]][c], in f64, plus sum |weight * out| per output for the error model.
 */
void orc_moe_combine(const float *out, const int32_t *pair_rows, const float *weights,
                     int64_t T, int topk, int64_t n, double *y, double *absy)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < n; ++c) {
            double acc = 0.0, aabs = 0.0;
            for (int j = 0; j < topk; ++j) {
                const double term = (double)weights[t * topk + j] *
                                    (double)out[(int64_t)pair_rows[t * topk + j] * n + c];
                acc += term;
                aabs += fabs(term);
            }
            y[t * n + c] = acc;
            absy[t * n + c] = aabs;
        }
}

/* ------------------------------------------------------------------ W4A4 [W] */

uint8_t orc_e2m1_encode(float v)
{
    /* Nearest E2M1 magnitude by exhaustive search over the eight non-negative codes (their
     * values increase with the code); on a tie the even code wins. Magnitudes of 6 and
     * above saturate to 6 (code 7) directly: far above 6 every distance rounds alike. */
    init_tables();
    const int neg = signbit(v) ? 1 : 0;
    const double a = fabs((double)v);
    if (a >= 6.0)
        return (uint8_t)(7 | (neg ? 0x8 : 0x0));
    int best = 0;
    double bestd = a - g_e2m1[0];
    for (int c = 1; c < 8; ++c) {
        const double d = fabs(a - g_e2m1[c]);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) != 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(best | (neg ? 0x8 : 0x0));
}

/* Quantise the 16 values v[0..15] against the micro-scale of e4m3 code s into codes16
 * (one nibble per value, unpacked). */
static void e2m1_block(const float *v, uint8_t s, uint8_t *codes16)
{
    const float S = (float)g_e4m3[s];
    for (int i = 0; i < 16; ++i)
        codes16[i] = S == 0.0f ? 0 : orc_e2m1_encode(v[i] / S);
}

static void pack_nibbles(const uint8_t *codes16, uint8_t *dst8)
{
    for (int i = 0; i < 8; ++i)
        dst8[i] = (uint8_t)(codes16[2 * i] | (codes16[2 * i + 1] << 4));
}

void orc_act_quant_w4a4(const float *x, int64_t rows, int64_t k, uint8_t *codes, uint8_t *scales,
                        float *rowscale)
{
    init_tables();
    const int64_t nb = k / 16;
    for (int64_t r = 0; r < rows; ++r) {
        const float *row = x + r * k;
        float amax = 0.0f;
        for (int64_t i = 0; i < k; ++i)
            if (fabsf(row[i]) > amax)
                amax = fabsf(row[i]);
        const float rs = amax / 2688.0f; /* 6 * 448 */
        rowscale[r] = rs;
        for (int64_t j = 0; j < nb; ++j) {
            float y[16];
            uint8_t c16[16];
            uint8_t s = 0;
            if (rs != 0.0f) {
                float m = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    y[i] = row[j * 16 + i] / rs;
                    if (fabsf(y[i]) > m)
                        m = fabsf(y[i]);
                }
                s = orc_e4m3_encode(m / 6.0f);
                e2m1_block(y, s, c16);
            } else {
                memset(c16, 0, sizeof c16);
            }
            scales[r * nb + j] = s;
            pack_nibbles(c16, codes + r * (k / 2) + j * 8);
        }
    }
}

void orc_act_quant_w4a4_v1(const float *x, int64_t rows, int64_t k, uint8_t *codes,
                           uint8_t *scales)
{
    init_tables();
    const int64_t nb = k / 16;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < nb; ++j) {
            const float *v = x + r * k + j * 16;
            float m = 0.0f;
            for (int i = 0; i < 16; ++i)
                if (fabsf(v[i]) > m)
                    m = fabsf(v[i]);
            uint8_t s = orc_e4m3_encode(m / 6.0f);
            if (s == 0 && m > 0.0f)
                s = 0x01;
            uint8_t c16[16];
            e2m1_block(v, s, c16);
            scales[r * nb + j] = s;
            pack_nibbles(c16, codes + r * (k / 2) + j * 8);
        }
    }
}

void orc_gemm_ref_w4a4(const uint8_t *codes, const uint8_t *scales, const float *rowscale,
                       const uint8_t *w, const uint8_t *sc, float scale2, int64_t g, int64_t n,
                       int64_t k, double *out, double *absp)
{
    init_tables();
    const int64_t nb = k / 16;
    for (int64_t row = 0; row < g; ++row) {
        const double rs = rowscale ? (double)rowscale[row] : 1.0;
        const double outer = rs * (double)scale2;
        for (int64_t col = 0; col < n; ++col) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t j = 0; j < nb; ++j) {
                const double sa = g_e4m3[scales[row * nb + j]];
                const double sw = g_e4m3[sc[col * nb + j]];
                for (int i = 0; i < 16; ++i) {
                    const int64_t kk = j * 16 + i;
                    const uint8_t ab = codes[row * (k / 2) + (kk >> 1)];
                    const uint8_t wb = w[col * (k / 2) + (kk >> 1)];
                    const uint8_t an = (kk & 1) ? (uint8_t)(ab >> 4) : (uint8_t)(ab & 0x0F);
                    const uint8_t wn = (kk & 1) ? (uint8_t)(wb >> 4) : (uint8_t)(wb & 0x0F);
                    const double p = g_e2m1[an] * sa * g_e2m1[wn] * sw * outer;
                    acc += p;
                    aabs += fabs(p);
                }
            }
            out[row * n + col] = acc;
            absp[row * n + col] = aabs;
        }
    }
}
