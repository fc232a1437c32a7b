// internal.h -- declarations shared by the library's translation units (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "fp4moe.h"  // include/ is on the compiler include path

namespace fp4moe {

// One grouped projection as the kernels see it. Single-expert calls use E = 1 and
// offsets == nullptr (rows [0, P)).
struct GroupedProblem {
    const float *x;          // [T, k] f32
    int64_t T;               // rows of x
    const int32_t *row_ids;  // nullable [P]
    const int32_t *offsets;  // nullable [E+1] (device)
    int E;
    int64_t P;               // routed rows
    const uint8_t *w;        // [E, n, k/2]
    const uint8_t *sc;       // [E, n, k/gs]
    const float *scale2;     // nullable [E] (device)
    float scale2_host;       // used when scale2 == nullptr (NVFP4)
    int recipe;              // FP4_NVFP4 / FP4_MXFP4
    float *out;              // [P, n]
    int n;
    int k;
    uint8_t *codes_out;      // nullable [P, k]  (single-expert calls)
    float *scales_out;       // nullable [P, k/128]
    unsigned *err;           // device error word of the current device
};

// Address of the current device's error word (looked up once per device).
unsigned *device_error_word();

// Fused SwiGLU output of a gate/up projection on the tensor-core path: the bank holds
// 2 inter rows per expert (gate rows, then up rows) and the call writes
// h = SwiGLU(gate, up) with the swiglu_limit clamps, [P, inter] f32, instead of [P, 2 inter].
struct SwigluOut {
    float *h;
    int64_t inter;  // a multiple of 64
    float limit;
};

// The tensor-core path (gemm_tc.cu: NVFP4 on the 16-bit MMA; gemm_mx.cu: MXFP4 on the
// block-scaled 8-bit MMA): workspace size, shape support, the quantise phase and the GEMM.
size_t tc_workspace_bytes(int64_t num_tokens, int64_t total_rows, int64_t k, int recipe);
bool tc_supported(int64_t n, int64_t k, int recipe, int E);
cudaError_t launch_tc_quantize(const GroupedProblem &p, void *workspace, cudaStream_t s);
cudaError_t launch_tc_gemm(const GroupedProblem &p, const void *workspace, cudaStream_t s,
                           const SwigluOut *sw = nullptr);
size_t mx_workspace_bytes(int64_t num_tokens, int64_t total_rows, int64_t k);
bool mx_supported(int64_t n, int64_t k, int E, const void *w);
cudaError_t launch_mx_quantize(const GroupedProblem &p, void *workspace, cudaStream_t s);
cudaError_t launch_mx_gemm(const GroupedProblem &p, const void *workspace, cudaStream_t s,
                           const SwigluOut *sw = nullptr);

// The W4A4 variant (gemm_w4a4.cu): two-level E2M1 activations against NVFP4 weights on
// the block-scaled 4-bit MMA. w4a4_supported: the shapes the GEMM takes (k % 256 == 0, at
// most 1024 experts); its weight and scale bases must also be 16-byte aligned.
// launch_act_quant_w4a4 quantises S source rows (x[rid[s]] or x[s]).
size_t w4a4_workspace_bytes(int64_t num_tokens, int64_t total_rows, int64_t k);
bool w4a4_supported(int64_t n, int64_t k, int E);
cudaError_t launch_act_quant_w4a4(const float *x, const int32_t *rid, int64_t T, int64_t S,
                                  int64_t k, uint8_t *codes, uint8_t *scales, float *rowscale,
                                  unsigned *err, cudaStream_t s);
cudaError_t launch_w4a4_quantize(const GroupedProblem &p, void *workspace, cudaStream_t s);
cudaError_t launch_w4a4_gemm(const GroupedProblem &p, const void *workspace, cudaStream_t s);

// The bounded-wait limit (clock64 cycles) for the next tensor-core GEMM launch on this host
// thread. Sets *stall to 1 and clears the request if fp4_test_stall_next_gemm asked for a
// stalled launch; otherwise returns the normal limit and leaves *stall alone.
long long take_stall_request(int *stall);

// Kernel launchers; each returns cudaSuccess or the launch error.
cudaError_t launch_act_quant(const float *x, uint8_t *codes, float *scales, int64_t rows,
                             int64_t k, cudaStream_t s);
cudaError_t launch_mirror_gemm(const uint8_t *codes, const float *scales, const uint8_t *w,
                               const uint8_t *wscale, float scale2, int recipe, float *out,
                               int64_t g, int64_t n, int64_t k, cudaStream_t s);
cudaError_t launch_swiglu_quant(const float *gate, const float *up, int64_t ld, float limit,
                                int64_t rows, int64_t inter, float *h_out, uint8_t *codes,
                                float *scales, cudaStream_t s);
cudaError_t launch_stream_gemm(const GroupedProblem &p, int rows_per_pass, cudaStream_t s);
// Decode kernel (warp-level MMA); rows_per_pass 4 or 8 (8 only where they fit).
// decode_fits(k): its shared memory holds 4 activation rows of length k (k <= 28544).
cudaError_t launch_decode_gemm(const GroupedProblem &p, int rows_per_pass, cudaStream_t s);
bool decode_fits(int64_t k);

// Routing front-end (routing.cu).
cudaError_t launch_route_topk(const float *logits, int64_t T, int E, int topk, int renormalize,
                              int32_t *ids, float *weights, cudaStream_t s);
size_t route_csr_workspace_bytes(int64_t T, int E);
cudaError_t launch_route_csr(const int32_t *ids, int64_t T, int topk, int E, int32_t *offsets,
                             int32_t *row_ids, int32_t *pair_rows, void *workspace,
                             unsigned *err, cudaStream_t s);
cudaError_t launch_moe_combine(const float *out, const int32_t *pair_rows, const float *weights,
                               int64_t T, int topk, int64_t n, int64_t P, float *y, unsigned *err,
                               cudaStream_t s);

// Error-model constants of each path (n_ops of |err| <= n_ops 2^-24 sum|p|).
double stream_error_ops(int recipe, int64_t k);
double decode_error_ops(int recipe, int64_t k);

} // namespace fp4moe
