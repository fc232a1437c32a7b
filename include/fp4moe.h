/*
 * fp4moe.h -- C ABI of libfp4moe.so: the quantized MoE expert projection on GB300 (sm_103a).
 *
 * The operation (memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs):
 *   1. fn quant_rows: every activation row is cut into groups of 128; per group
 *      amax = max(max|x|, 1e-4), s = pow2_ceil(amax * f32(1/448)) and
 *      code = e4m3(clamp(x / s, -448, 448)) (round to nearest even, sign kept).
 *   2. fn f64_ref / fn mirror_gemm: out[r][c] = sum over weight groups j of
 *      (sum_{i<gs} e4m3(code) * E2M1(nibble)) * (ws_j * s_{r, j*gs/128}), f32 accumulation,
 *      where NVFP4 (gs = 16) has ws = f32(e4m3(scale byte) * scale2) and MXFP4 (gs = 32)
 *      has ws = 2^(e8m0 byte - 127). Weight rows hold k/2 bytes of nibble pairs, the low
 *      nibble being the even k (struct ExpertRaw; the nibble split in mirror_gemm).
 *
 * Conventions for every call:
 *   - All array arguments are device pointers on the current CUDA device, row-major and
 *     contiguous, owned by the caller; the library allocates nothing and never frees.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are stream-ordered
 *     and asynchronous: they enqueue kernels and return without synchronising.
 *   - Sizes are elements unless named *_bytes. k must be a positive multiple of 128.
 *   - Every pointer must be 16-byte aligned (the kernels use 128-bit accesses).
 *   - The return value is an fp4_status; a non-zero status means nothing was enqueued.
 *   - Inputs must be finite: non-finite activations give unspecified codes (no crash).
 *   - Device-side checks (CSR offsets, row ids) cannot return a status without a sync;
 *     they set bits in a per-device error word read by fp4_get_device_error().
 */
#ifndef FP4MOE_H
#define FP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP4_OK = 0,
    FP4_ERR_ARG = -1,       /* null required pointer, unknown recipe, negative size */
    FP4_ERR_SHAPE = -2,     /* k % 128 != 0, k or n < 1, sizes past the supported range */
    FP4_ERR_ALIGN = -3,     /* a pointer that is not 16-byte aligned */
    FP4_ERR_LAUNCH = -4,    /* the CUDA runtime refused a launch (see fp4_last_error) */
    FP4_ERR_DEVICE = -5,    /* returned by fp4_get_device_error when device checks failed */
    FP4_ERR_WORKSPACE = -6  /* workspace missing or below fp4_grouped_workspace_size() */
} fp4_status;

typedef enum { FP4_NVFP4 = 0, FP4_MXFP4 = 1 } fp4_recipe; /* matches the pages' kind 0/1 */

/* Bits of the device error word (fp4_get_device_error). */
enum {
    FP4_DEVERR_OFFSETS = 1, /* offsets not non-decreasing from 0 to total_rows */
    FP4_DEVERR_ROW_ID = 2,  /* a row id outside [0, num_tokens) */
    FP4_DEVERR_TIMEOUT = 4,  /* a pipeline wait gave up after its iteration limit */
    FP4_DEVERR_EXPERT_ID = 8 /* an expert id outside [0, num_experts) or repeated in a token */
};

/* Kernel paths (fp4_gemm_path / fp4_force_path). */
enum {
    FP4_PATH_AUTO = 0,   /* library choice by shape (fp4_gemm_path) */
    FP4_PATH_STREAM = 1, /* no-workspace weight streaming with a fused act-quant prologue:
                            warp-level MMA (mma.sync) for k <= 28544, CUDA-core FMA above */
    FP4_PATH_TC = 2      /* tcgen05 tensor-core kernel over a quantized-activation workspace */
};

/*
 * act_quant_fp8 -- stage 1 alone (fn quant_rows of dsv4_native_gemm_gate.rs).
 *   x      [rows, k] f32 in
 *   codes  [rows, k] e4m3 bytes out
 *   scales [rows, k/128] f32 out (powers of two)
 * Bit-exact with the oracle's act_quant. rows == 0 is a no-op returning FP4_OK.
 */
int act_quant_fp8(const float *x, uint8_t *codes, float *scales, int64_t rows, int64_t k,
                  void *stream);

/*
 * fp4_expert_gemm -- one expert, act_quant fused into the GEMM:
 * out[g, n] = quant(x)[g, k] . W[n, k]^T (fn f64_ref / fn mirror_gemm of
 * dsv4_native_gemm_gate.rs, with the activation quantized on device first).
 *   x          [g, k] f32 activations
 *   w          [n, k/2] nibble pairs (low nibble = even k)
 *   wscale     [n, k/16] e4m3 bytes (NVFP4) or [n, k/32] e8m0 bytes (MXFP4)
 *   scale2     per-tensor f32 factor (NVFP4; ignored for MXFP4)
 *   out        [g, n] f32
 *   codes_out  nullable [g, k] e4m3 bytes: the quantized activations (as act_quant_fp8)
 *   scales_out nullable [g, k/128] f32
 *   workspace  nullable; with at least fp4_grouped_workspace_size(g, g, n, k, recipe)
 *              bytes the tensor-core path may be used, otherwise the streaming path.
 * Asking for codes_out costs nothing on the streaming path (its prologue quantises
 * anyway) and one extra act_quant pass over x on the tensor-core path.
 */
int fp4_expert_gemm(const float *x, const uint8_t *w, const uint8_t *wscale, float scale2,
                    int recipe, float *out, int64_t g, int64_t n, int64_t k, uint8_t *codes_out,
                    float *scales_out, void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes fp4_grouped_expert_gemm (and fp4_expert_gemm) needs for this shape. */
size_t fp4_grouped_workspace_size(int64_t num_tokens, int64_t total_rows, int64_t n, int64_t k,
                                  int recipe);

/*
 * fp4_grouped_expert_gemm -- all experts of one projection in one call. Routed row p
 * (0 <= p < total_rows) reads activation row x[row_ids[p]] (x[p] when row_ids is NULL)
 * and belongs to the expert e with offsets[e] <= p < offsets[e+1] (CSR offsets, as the
 * grouped MoE GEMM section of memra-engine 0.71.0 src/bin/kernel_check.rs builds them).
 *   x         [num_tokens, k] f32
 *   row_ids   nullable [total_rows] int32 (device)
 *   offsets   [num_experts + 1] int32 (device): offsets[0] = 0, non-decreasing,
 *             offsets[num_experts] = total_rows
 *   w         [num_experts, n, k/2] nibble pairs; expert e's block starts at e*n*k/2
 *   wscale    [num_experts, n, k/gs] scale bytes
 *   scale2    [num_experts] f32 (device; NVFP4; may be NULL for MXFP4)
 *   out       [total_rows, n] f32
 *   workspace at least fp4_grouped_workspace_size(...) bytes (may be NULL if that is 0)
 * Experts with no rows cost nothing but a CTA exit. Offsets or row ids that fail the
 * device checks set fp4_get_device_error bits; their rows are skipped (out untouched).
 * Stream order is kept. The weight-streaming kernel is launched with programmatic stream
 * serialization: it may be scheduled while the kernel before it on the stream is still
 * draining, and it reads no global memory (inputs included) until that kernel has
 * completed, so any input may be the previous kernel's output.
 */
int fp4_grouped_expert_gemm(const float *x, int64_t num_tokens, const int32_t *row_ids,
                            const int32_t *offsets, int num_experts, int64_t total_rows,
                            const uint8_t *w, const uint8_t *wscale, const float *scale2,
                            int recipe, float *out, int64_t n, int64_t k, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * The tensor-core path of fp4_grouped_expert_gemm in its two halves, for callers that
 * time them apart or run several projections over one quantised input (the gate and up
 * banks of one x, say). fp4_grouped_expert_gemm with a workspace on that path is exactly
 * fp4_grouped_quantize followed by fp4_grouped_gemm_quantized on the same stream.
 *
 * fp4_grouped_quantize -- stage 1 (fn quant_rows of dsv4_native_gemm_gate.rs) written into
 * the workspace as the operands of the tensor-core GEMM. NVFP4: the 16-bit operands
 * f16(code * 2^(m - M)) with a per-row power-of-two scale 2^M (while every 128-block of the
 * row lies within 2^15 of its largest) or bf16(code * 2^m) (calls with a wider row), both
 * exact. MXFP4: the e4m3 codes themselves and each block's scale exponent as a byte (the
 * block-scaled 8-bit MMA's own operand and scale formats). When row ids repeat tokens (row_ids given and num_tokens < total_rows) each
 * token row is quantised once and the result copied to its routed rows; otherwise every
 * routed row x[row_ids[p]] (x[p]) is quantised. The workspace layout is private to the
 * library.
 *   x, num_tokens, row_ids, total_rows, k, recipe: as fp4_grouped_expert_gemm
 *   workspace at least fp4_grouped_workspace_size(num_tokens, total_rows, n, k, recipe) bytes
 * Row ids outside [0, num_tokens) set FP4_DEVERR_ROW_ID; such rows quantise as zeros.
 * Shapes the tensor-core path does not take (k not a multiple of 16*gs) return
 * FP4_ERR_SHAPE.
 */
int fp4_grouped_quantize(const float *x, int64_t num_tokens, const int32_t *row_ids,
                         int64_t total_rows, int64_t k, int recipe, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * fp4_grouped_gemm_quantized -- stage 2 on the tensor cores (fn f64_ref of
 * dsv4_native_gemm_gate.rs, f32 accumulation) from a workspace that fp4_grouped_quantize
 * filled earlier on the same stream for the same num_tokens, row ids, total_rows, k and
 * recipe; the workspace is only read, so one quantised input serves any number of these
 * calls. (Row ids are checked by fp4_grouped_quantize: outside [0, num_tokens) they set
 * FP4_DEVERR_ROW_ID and give zero rows.)
 *   num_tokens, row_ids, offsets, num_experts, w, wscale, scale2, out, n: as
 *   fp4_grouped_expert_gemm
 * Always the tensor-core path (whatever the rows per expert); error model
 * fp4_error_ops(FP4_PATH_TC, recipe, k).
 */
int fp4_grouped_gemm_quantized(const void *workspace, size_t workspace_bytes,
                               int64_t num_tokens, const int32_t *row_ids,
                               const int32_t *offsets, int num_experts, int64_t total_rows,
                               const uint8_t *w, const uint8_t *wscale, const float *scale2,
                               int recipe, float *out, int64_t n, int64_t k, void *stream);

/*
 * fp4_grouped_expert_gemm_noalloc -- the same computation as fp4_grouped_expert_gemm,
 * on the tensor-core path, for callers that cannot allocate device memory (a host
 * framework that owns all device memory and forbids libraries to allocate, a serving
 * loop with a no-allocation rule after start-up, or code where an allocation would
 * synchronise the device at the wrong time). It takes no workspace: its scratch is a
 * fixed 32 MiB device array inside this library, which every GPU that loads the library
 * holds until the process exits. The pages have no counterpart of this call.
 *   Arguments: as fp4_grouped_expert_gemm without workspace/workspace_bytes.
 *   Limit: the call needs fp4_grouped_workspace_size(num_tokens, total_rows, n, k, recipe)
 *          bytes of scratch, at most 32 MiB: for NVFP4 2048 + R(2 * total_rows * k) +
 *          R(4 * total_rows), plus R(2 * num_tokens * k) + R(4 * num_tokens) when
 *          num_tokens < total_rows; for MXFP4 1024 + R(total_rows * k) +
 *          R(k/128 * P16(total_rows)), plus R(num_tokens * k) + R(k/128 * P16(num_tokens))
 *          when num_tokens < total_rows (R rounds up to a multiple of 1024, P16 to a
 *          multiple of 16) (e.g. 2048 routed rows at k = 7168, or 2048
 *          routed rows of 256 tokens); larger calls return
 *          FP4_ERR_WORKSPACE (the message in fp4_last_error gives both numbers), shapes the
 *          tensor-core path does not take (k not a multiple of 16*gs, more than 1024
 *          experts) return FP4_ERR_SHAPE. The call itself allocates, frees and synchronises
 *          nothing.
 *   First call on a device: looks up the scratch array's device address for that
 *          device (cudaGetSymbolAddress), so make it before any stream capture. The
 *          driver reserves the array when this library's device code is first loaded on
 *          a device (at the first call that needs it under lazy module loading, or when
 *          the library is loaded with eager loading), and that reservation may
 *          synchronise: make one warm-up call per device before any phase in which
 *          nothing may allocate or synchronise.
 *   Sharing: every call uses the same array and leaves its contents behind; nothing in
 *          it needs to start at zero. Calls whose kernels overlap on the GPU (other
 *          streams, other threads) race on it: serialise them.
 */
int fp4_grouped_expert_gemm_noalloc(const float *x, int64_t num_tokens, const int32_t *row_ids,
                                    const int32_t *offsets, int num_experts, int64_t total_rows,
                                    const uint8_t *w, const uint8_t *wscale, const float *scale2,
                                    int recipe, float *out, int64_t n, int64_t k, void *stream);

/*
 * fp4_gemm_mirror -- one expert's GEMM from already-quantised activations, in the page's
 * own kernel order (dsv4_native_gemm_gate.rs, fn mirror_gemm), bit for bit: per output,
 * 128 partials (partial t takes weight groups t, t+128, ...; a group's gs products summed
 * in k order, times f32(ws * as), added), then a fixed halving tree; every operation a
 * separately rounded f32 multiply or add. Arguments as the page's memra_dsv4_fp4_gemm:
 *   codes  [g, k] e4m3 bytes, scales [g, k/128] f32 (as act_quant_fp8 writes them)
 *   w      [n, k/2] nibble pairs, wscale [n, k/gs] scale bytes, scale2 (NVFP4)
 *   out    [g, n] f32
 * An instrument for bit-identity with the pages' mirror, not a fast path (one 128-thread
 * CTA per output). k must be a positive multiple of 128; g == 0 is a no-op.
 */
int fp4_gemm_mirror(const uint8_t *codes, const float *scales, const uint8_t *w,
                    const uint8_t *wscale, float scale2, int recipe, float *out, int64_t g,
                    int64_t n, int64_t k, void *stream);

/*
 * fp4_swiglu_quant -- the step after the gate/up projection: SwiGLU with the
 * swiglu_limit clamps (dsv4_native_gemm_gate.rs, swiglu_limit saturation cell and the f64
 * check of main), fused with fn quant_rows of its output (the down projection's input):
 *   u = clamp(up, -limit, limit), g = min(gate, limit), h = g * (1 / (1 + exp(-g))) * u,
 *   then per 128 elements of h: pow2 scale and e4m3 codes exactly as act_quant_fp8.
 *   gate, up  rows of `inter` f32 at a row stride of `ld` elements (ld >= inter,
 *             ld % 4 == 0): separate [rows, inter] tensors (ld = inter), or the two halves
 *             of a fused gate/up output [rows, 2*inter] (up = gate + inter, ld = 2*inter)
 *   limit     the swiglu_limit, finite and > 0
 *   h_out     nullable [rows, inter] f32: h itself (within a few ulps of exact: expf)
 *   codes     [rows, inter] e4m3 bytes, scales [rows, inter/128] f32 (powers of two);
 *             equal, bit for bit, to act_quant_fp8 of the h this call computed
 * inter must be a positive multiple of 128; rows == 0 is a no-op returning FP4_OK.
 * Inputs are finite (as everywhere in this library).
 */
int fp4_swiglu_quant(const float *gate, const float *up, int64_t ld, float limit, int64_t rows,
                     int64_t inter, float *h_out, uint8_t *codes, float *scales, void *stream);

/*
 * fp4_grouped_gate_up_swiglu -- the gate/up projection with SwiGLU in its epilogue: the
 * grouped call of fp4_grouped_expert_gemm over a gate/up bank, writing
 * h = SwiGLU(gate, up) with the swiglu_limit clamps (the arithmetic of fp4_swiglu_quant,
 * dsv4_native_gemm_gate.rs swiglu_limit saturation cell) instead of the [P, 2*inter]
 * gate/up output. The down projection then takes h as its input rows
 * (fp4_grouped_expert_gemm with row_ids = NULL), whose own quantise pass is the page's
 * requantisation of h. Tensor-core path only.
 *   w, wscale  a gate/up bank [E, 2*inter, k/2], [E, 2*inter, k/gs]: rows [0, inter) of
 *              an expert are its gate rows, rows [inter, 2*inter) its up rows (the page's
 *              layout of w1 and w3 stacked)
 *   h          [total_rows, inter] f32 out, in routed-row order; every element equals,
 *              bit for bit, fp4_swiglu_quant's h of this call's gate/up output
 *   inter      a multiple of 64; workspace: fp4_grouped_workspace_size(num_tokens,
 *              total_rows, 2*inter, k, recipe) bytes
 * Other arguments and checks as fp4_grouped_expert_gemm; shapes the tensor-core path does
 * not take return FP4_ERR_SHAPE (use fp4_grouped_expert_gemm and fp4_swiglu_quant then).
 */
int fp4_grouped_gate_up_swiglu(const float *x, int64_t num_tokens, const int32_t *row_ids,
                               const int32_t *offsets, int num_experts, int64_t total_rows,
                               const uint8_t *w, const uint8_t *wscale, const float *scale2,
                               int recipe, float swiglu_limit, float *h, int64_t inter,
                               int64_t k, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The routing front-end: the steps before and after the grouped projections.
 *
 * fp4_route_topk -- the router (memra-engine 0.125.0, src/bin/qwen4exp_gpu_gate.rs,
 * device-router arm: a softmax top-k whose selected ids and their order are exact and
 * whose weights are within a few ulps; the pages do not print its body). Reading taken:
 * each token selects the topk experts with the largest logits, equal logits ranking the
 * lower expert id first, emitted best first; weights are softmax probabilities
 * exp(l - max) / sum over all experts, or with renormalize != 0 over the selected ones.
 *   logits  [num_tokens, num_experts] f32 (finite), 1 <= num_experts <= 1024
 *   ids     [num_tokens, topk] int32 out, weights [num_tokens, topk] f32 out
 *   1 <= topk <= min(32, num_experts)
 */
int fp4_route_topk(const float *logits, int64_t num_tokens, int num_experts, int topk,
                   int renormalize, int32_t *ids, float *weights, void *stream);

/* Workspace bytes fp4_route_csr needs (a bitmap and popcount prefix of num_experts x
 * ceil(num_tokens/32) words, and the experts' row counts). */
size_t fp4_route_csr_workspace_size(int64_t num_tokens, int num_experts);

/*
 * fp4_route_csr -- the CSR layout the grouped calls take (memra-engine 0.71.0,
 * src/bin/kernel_check.rs, grouped MoE GEMM section: offsets[e+1] = offsets[e] + rows of
 * expert e), built on the device from each token's expert ids. Routed rows are grouped by
 * expert and, within an expert, in token order; the result does not depend on thread
 * timing.
 *   ids        [num_tokens, topk] int32 (distinct within a token, in [0, num_experts))
 *   offsets    [num_experts + 1] int32 out (offsets[num_experts] = num_tokens * topk)
 *   row_ids    [num_tokens * topk] int32 out: the token of each routed row
 *   pair_rows  nullable [num_tokens, topk] int32 out: the routed row of each (token, slot)
 *   workspace  at least fp4_route_csr_workspace_size(num_tokens, num_experts) bytes
 * An id outside [0, num_experts) or repeated within a token sets FP4_DEVERR_EXPERT_ID;
 * the outputs are then unspecified.
 */
int fp4_route_csr(const int32_t *ids, int64_t num_tokens, int topk, int num_experts,
                  int32_t *offsets, int32_t *row_ids, int32_t *pair_rows, void *workspace,
                  size_t workspace_bytes, void *stream);

/*
 * fp4_moe_combine -- the weighted combine of the routed rows' outputs back to tokens
 * (memra-engine 0.71.0, src/bin/kernel_check.rs, grouped MoE GEMM section: a per-routed-
 * row factor on the output, summed here over a token's routed rows):
 *   y[t][c] = sum over slots j = 0 .. topk-1, in order, of weights[t][j] * out[pair_rows[t][j]][c]
 * with one f32 fma per slot (error model: n_ops = topk against the f64 sum of |terms|).
 *   out        [total_rows, n] f32 (a grouped call's output)
 *   pair_rows  [num_tokens, topk] int32 (from fp4_route_csr); rows outside
 *              [0, total_rows) set FP4_DEVERR_ROW_ID and are skipped
 *   weights    [num_tokens, topk] f32
 *   y          [num_tokens, n] f32 out; n must be a multiple of 4
 */
int fp4_moe_combine(const float *out, int64_t total_rows, const int32_t *pair_rows,
                    const float *weights, int64_t num_tokens, int topk, int64_t n, float *y,
                    void *stream);

/*
 * ---------------------------------------------------------------- W4A4 NVFP4 variant
 * E2M1 (4-bit) activations against NVFP4 weights (memra-engine 0.71.0,
 * src/bin/kernel_check.rs, the NVFP4 W4A4 MMQ GEMM section): a different numeric class
 * from the calls above (the activations lose far more than e4m3 codes do; the section
 * treats rel ~ 0.1 against the unquantised activations as normal). Two-level scaling, in
 * the reading this library takes (the page names the two levels, not the formulas):
 *   r = amax_row / 2688 (f32; 2688 = 6 * 448)      the per-token row scale
 *   y = x / r                                       (f32)
 *   s = e4m3 nearest to (max|y| over 16 values) / 6 the micro-scale, ties to the even code
 *   code = E2M1 nearest to y / S (S = value of s)   ties to the even code, |.| >= 6 -> 6,
 *                                                   sign kept; all zero where S = 0
 * A zero row has r = 0 and zero codes and scales. The GEMM then computes, on the
 * block-scaled 4-bit tensor cores (one e4m3 scale per 16 k on each operand, f32
 * accumulation),
 *   out[p][c] = (sum_k E2M1(a) S_a * E2M1(w) S_w) * r_p * scale2[e]
 * with every product exact; error model fp4_w4a4_error_ops(k) against the f64 sum over the
 * dequantised operands. The weight scale bytes must be non-negative e4m3 (sign bit clear:
 * the MMA reads them unsigned); NVFP4 scales are.
 *
 * act_quant_w4a4 -- the quantisation alone.
 *   x        [rows, k] f32 in; k a positive multiple of 16
 *   codes    [rows, k/2] out: E2M1 nibble pairs (low nibble = even k, as the weights)
 *   scales   [rows, k/16] out: micro-scale e4m3 bytes
 *   rowscale [rows] f32 out: r
 * All four pointers 16-byte aligned device memory owned by the caller. Bit-exact with the
 * oracle. rows == 0 is a no-op.
 */
int act_quant_w4a4(const float *x, uint8_t *codes, uint8_t *scales, float *rowscale, int64_t rows,
                   int64_t k, void *stream);

/* Workspace bytes the W4A4 grouped calls need (0 for shapes they do not take):
 * 1024 + R(P k/2) + R(P k/16) + R(4 P), plus R(T k/2) + R(T k/16) + R(4 T) when
 * num_tokens T < total_rows P (R rounds up to a multiple of 1024). */
size_t fp4_w4a4_workspace_size(int64_t num_tokens, int64_t total_rows, int64_t k);

/*
 * fp4_grouped_expert_gemm_w4a4 -- all experts of one NVFP4 projection with W4A4
 * activations, in one call (routing as fp4_grouped_expert_gemm: routed row p reads
 * x[row_ids[p]], or x[p] without row ids, and belongs to the expert e with
 * offsets[e] <= p < offsets[e+1]).
 *   x, num_tokens, row_ids, offsets, num_experts, total_rows: as fp4_grouped_expert_gemm
 *   w        [num_experts, n, k/2] nibble pairs, 16-byte aligned
 *   wscale   [num_experts, n, k/16] e4m3 bytes (non-negative), 16-byte aligned
 *   scale2   [num_experts] f32 (device)
 *   out      [total_rows, n] f32
 *   workspace at least fp4_w4a4_workspace_size(num_tokens, total_rows, k) bytes
 * k must be a multiple of 256 and num_experts at most 1024 (else FP4_ERR_SHAPE). When row
 * ids repeat tokens (num_tokens < total_rows) each token row is quantised once and copied
 * to its routed rows. Offsets or row ids that fail the device checks set
 * fp4_get_device_error bits (bad row ids give zero rows; bad offsets skip the call's rows).
 * Always the tensor-core kernel, at any number of rows per expert.
 */
int fp4_grouped_expert_gemm_w4a4(const float *x, int64_t num_tokens, const int32_t *row_ids,
                                 const int32_t *offsets, int num_experts, int64_t total_rows,
                                 const uint8_t *w, const uint8_t *wscale, const float *scale2,
                                 float *out, int64_t n, int64_t k, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* fp4_grouped_expert_gemm_w4a4 in its two halves (the quantise pass into the workspace,
 * then the GEMM that only reads it), for callers that time them apart or run several
 * projections over one quantised input. Arguments as fp4_grouped_expert_gemm_w4a4; the
 * workspace of fp4_w4a4_gemm_quantized must have been filled by fp4_w4a4_quantize on the
 * same stream for the same num_tokens, row ids, total_rows and k. */
int fp4_w4a4_quantize(const float *x, int64_t num_tokens, const int32_t *row_ids,
                      int64_t total_rows, int64_t k, void *workspace, size_t workspace_bytes,
                      void *stream);
int fp4_w4a4_gemm_quantized(const void *workspace, size_t workspace_bytes, int64_t num_tokens,
                            const int32_t *row_ids, const int32_t *offsets, int num_experts,
                            int64_t total_rows, const uint8_t *w, const uint8_t *wscale,
                            const float *scale2, float *out, int64_t n, int64_t k, void *stream);

/* n_ops of |out - f64 reference over the dequantised operands| <= n_ops 2^-24 sum|p| for
 * the W4A4 GEMM: k/16 + 3 (one rounding per 16-group of the f32 accumulation, as the other
 * tensor-core paths, plus the r and scale2 multiplies, plus one). Where r is so small that
 * those multiplies round in the f32 subnormal range (rows of subnormal inputs), each adds
 * up to 2^-150 absolute (gradual underflow): 2^-149 on top of the bound. */
double fp4_w4a4_error_ops(int64_t k);

/* Which path a grouped call of this shape takes (never FP4_PATH_AUTO): the tensor-core
 * path when a workspace is given, the shape is one it supports and the routed rows
 * average at least 9 per expert; the no-workspace path otherwise. */
int fp4_gemm_path(int64_t total_rows, int num_experts, int64_t n, int64_t k, int recipe,
                  int have_workspace);

/*
 * The n_ops of the per-output error model |out - f64 reference| <= n_ops * 2^-24 *
 * sum|scaled products| (dsv4_native_gemm_gate.rs, header comment and the f64 check)
 * for `path` at this recipe and k. Derived from the kernel's summation structure:
 * FP4_PATH_TC k/16 + 1 (+2 NVFP4); FP4_PATH_STREAM the same for k <= 28544 (the MMA
 * kernel), (gs-1) + 2*ceil(k/1024) (NVFP4; MXFP4 ceil(k/1024)) + 5 above (the FMA kernel).
 */
double fp4_error_ops(int path, int recipe, int64_t k);

/* Test hook: force a path for later calls made on the calling host thread (other threads
 * keep the choice by shape); FP4_PATH_AUTO restores the choice by shape. */
void fp4_force_path(int path);

/*
 * Test hook for the bounded-wait abort path (off unless called; the pages have no
 * counterpart: their calls report failure only through the status they return). The next
 * tensor-core GEMM launch made from the calling host thread (either recipe; it is the GEMM
 * phase of fp4_grouped_expert_gemm, fp4_grouped_gemm_quantized or the allocation-free
 * call) runs with one pipeline arrival withheld in its first CTA and with its waits bounded
 * by wait_limit_cycles clock64 cycles (clamped to [1e6, the normal limit of about 2e9]).
 * That launch gives up the stalled wait, sets FP4_DEVERR_TIMEOUT, drains its own copies
 * and MMAs, frees its tensor memory and returns; its outputs are unspecified. The request
 * is used once; wait_limit_cycles <= 0 withdraws it. Nothing faults or hangs.
 */
void fp4_test_stall_next_gemm(int64_t wait_limit_cycles);

/*
 * Synchronises `stream`, then returns FP4_OK or FP4_ERR_DEVICE and stores the device
 * error word (FP4_DEVERR_* bits) of the current device in *bits (nullable), clearing it.
 */
int fp4_get_device_error(void *stream, unsigned *bits);

/* Text of the last CUDA error a call met on this thread ("" if none). */
const char *fp4_last_error(void);

/* Name of a status code. */
const char *fp4_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FP4MOE_H */
