/*
 * oracle.h -- declarations of the CPU oracle (test infrastructure only; see oracle.c).
 * Nothing in the CUDA library includes this header.
 */
#ifndef FP4MOE_ORACLE_H
#define FP4MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_NVFP4 = 0, ORC_MXFP4 = 1 };

double orc_e4m3_decode(uint8_t b);
double orc_e2m1_decode(uint8_t nib);
double orc_e8m0_decode(uint8_t e);
uint8_t orc_e4m3_encode(float v);
float orc_pow2_ceil(float x);

/* x [rows,k] f32 -> codes [rows,k] e4m3 bytes, scales [rows,k/128] f32; k % 128 == 0. */
void orc_act_quant(const float *x, int64_t rows, int64_t k, uint8_t *codes, float *scales);

/* f64 reference: out/absp [g,n]; w [n,k/2] nibble pairs; sc [n,k/gs]. */
void orc_gemm_ref(const uint8_t *codes, const float *scales, const uint8_t *w, const uint8_t *sc,
                  float scale2, int recipe, int64_t g, int64_t n, int64_t k, double *out,
                  double *absp);

/* Grouped reference at sampled (routed row, column) pairs; samples sorted by row. */
int orc_grouped_ref_sampled(const float *x, int64_t T, int64_t k, const int32_t *row_ids,
                            const int32_t *offsets, int num_experts, int64_t P, const uint8_t *w,
                            const uint8_t *sc, const float *scale2, int recipe, int64_t n,
                            const int64_t *sample_p, const int64_t *sample_col, int64_t ns,
                            double *out, double *absp, uint8_t *tmp_codes, float *tmp_scales);

/* The page's mirror order in f32 (128 strided partials + halving tree): out [g,n]. */
void orc_mirror_gemm(const uint8_t *codes, const float *scales, const uint8_t *w,
                     const uint8_t *sc, float scale2, int recipe, int64_t g, int64_t n, int64_t k,
                     float *out);

/* SwiGLU with the swiglu_limit clamps, in f64: gate/up rows of stride ld (elements),
 * h [rows, inter]. */
void orc_swiglu(const float *gate, const float *up, int64_t ld, int64_t rows, int64_t inter,
                float limit, double *h);

/* Routing front-end: softmax top-k router (reading in oracle.c), CSR construction,
 * weighted combine of the routed rows' outputs back to tokens. */
void orc_route_topk(const float *logits, int64_t T, int E, int topk, int renormalize,
                    int32_t *ids, double *weights);
int orc_route_csr(const int32_t *ids, int64_t T, int topk, int E, int32_t *offsets,
                  int32_t *row_ids, int32_t *pair_rows);
void orc_moe_combine(const float *out, const int32_t *pair_rows, const float *weights,
                     int64_t T, int topk, int64_t n, double *y, double *absy);

/* W4A4 (two-level scaling; readings in oracle.c): x [rows,k] f32, k % 16 == 0 ->
 * codes [rows,k/2] nibble pairs (low nibble = even k), scales [rows,k/16] e4m3 bytes,
 * rowscale [rows] f32. The V1 form has no row scale. */
uint8_t orc_e2m1_encode(float v);
void orc_act_quant_w4a4(const float *x, int64_t rows, int64_t k, uint8_t *codes, uint8_t *scales,
                        float *rowscale);
void orc_act_quant_w4a4_v1(const float *x, int64_t rows, int64_t k, uint8_t *codes,
                           uint8_t *scales);
/* f64 reference of the W4A4 GEMM: out/absp [g,n]; rowscale nullable (1); w [n,k/2],
 * sc [n,k/16] e4m3 bytes, scale2 the weight tensor's factor. */
void orc_gemm_ref_w4a4(const uint8_t *codes, const uint8_t *scales, const float *rowscale,
                       const uint8_t *w, const uint8_t *sc, float scale2, int64_t g, int64_t n,
                       int64_t k, double *out, double *absp);

#ifdef __cplusplus
}
#endif

#endif
