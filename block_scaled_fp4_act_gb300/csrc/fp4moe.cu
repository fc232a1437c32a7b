// fp4moe.cu -- the exported C ABI (include/fp4moe.h): argument checks, path choice,
// kernel launches and the per-device error word. No allocation, no synchronisation in
// the compute calls.
#include <stdio.h>
#include <string.h>

#include "common.cuh"

namespace fp4moe {

__device__ unsigned int g_device_error = 0u;

unsigned *device_error_word()
{
    static unsigned *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    if (!addr[dev]) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_device_error) != cudaSuccess)
            return nullptr;
        addr[dev] = static_cast<unsigned *>(a);
    }
    return addr[dev];
}

int stream_max_rows_per_pass(int k);

// The tensor-core path by recipe: NVFP4 on the 16-bit MMA with converted weights, MXFP4 on
// the block-scaled 8-bit MMA (weights as stored, e4m3 activation codes).
static size_t tc_path_workspace(int64_t T, int64_t P, int64_t k, int recipe)
{
    return recipe == FP4_MXFP4 ? mx_workspace_bytes(T, P, k) : tc_workspace_bytes(T, P, k, recipe);
}

static cudaError_t tc_path_quantize(const GroupedProblem &p, void *ws, cudaStream_t s)
{
    return p.recipe == FP4_MXFP4 ? launch_mx_quantize(p, ws, s) : launch_tc_quantize(p, ws, s);
}

static cudaError_t tc_path_gemm(const GroupedProblem &p, const void *ws, cudaStream_t s,
                                const SwigluOut *sw = nullptr)
{
    return p.recipe == FP4_MXFP4 ? launch_mx_gemm(p, ws, s, sw) : launch_tc_gemm(p, ws, s, sw);
}

// Shapes (and, for MXFP4, the weight alignment the packed 4-bit TMA form needs) the
// tensor-core path takes.
static bool tc_path_supported(int64_t n, int64_t k, int recipe, int E, const void *w)
{
    if (!tc_supported(n, k, recipe, E))
        return false;
    return recipe != FP4_MXFP4 || mx_supported(n, k, E, w);
}
double tc_error_ops(int recipe, int64_t k);

// Path forced by fp4_force_path for calls made on the same host thread.
static thread_local int g_forced_path = FP4_PATH_AUTO;
// Wait limit of a stalled launch requested by fp4_test_stall_next_gemm (0: none).
static thread_local long long g_stall_limit = 0;

long long take_stall_request(int *stall)
{
    const long long limit = g_stall_limit;
    if (limit <= 0)
        return kTimeoutCycles;
    g_stall_limit = 0;
    *stall = 1;
    return limit;
}
static thread_local char g_last_error[256] = "";

static int record(cudaError_t e)
{
    if (e == cudaSuccess)
        return FP4_OK;
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
    return FP4_ERR_LAUNCH;
}

// Lets other translation units report a message through fp4_last_error.
void set_last_error(const char *msg)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

static bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u;
}

static bool recipe_ok(int r)
{
    return r == FP4_NVFP4 || r == FP4_MXFP4;
}

// Rows per expert (on average) at or above which the tensor-core path, workspace pass
// included, is faster than the warp-MMA decode kernel. Measured on GB300 (bench.py
// --path-sweep: 64 NVFP4 experts, [3072, 4096], L2 flushed): decode 107 / 117 / 193 us at
// 4 / 8 / 16 rows per expert, tensor cores 180 us throughout. The decode kernel streams
// the weights once per pass of up to 8 rows, so from 9 rows it streams them twice; the
// tensor-core kernel converts them once per 192-row tile.
constexpr int64_t kTcMinRowsPerExpert = 9;

static int choose_path(int64_t P, int E, int64_t n, int64_t k, int recipe, bool have_ws)
{
    const int forced = g_forced_path;
    if (forced != FP4_PATH_AUTO)
        return forced;
    if (have_ws && tc_supported(n, k, recipe, E) && P >= kTcMinRowsPerExpert * (int64_t)E)
        return FP4_PATH_TC;
    return FP4_PATH_STREAM;
}

// As choose_path, for a call whose weights are known (MXFP4 also needs them 32-byte aligned).
static int choose_path_for(const GroupedProblem &p, bool have_ws)
{
    const int path = choose_path(p.P, p.E, p.n, p.k, p.recipe, have_ws);
    if (path == FP4_PATH_TC && g_forced_path != FP4_PATH_TC &&
        !tc_path_supported(p.n, p.k, p.recipe, p.E, p.w))
        return FP4_PATH_STREAM;
    return path;
}

// The path that needs no workspace: the warp-MMA decode kernels wherever 4 activation rows
// of length k fit in shared memory (k <= 28544; 8 rows per pass where they fit and experts
// average more than 4): TMA-fed where k is a multiple of 512, per-lane loads otherwise;
// the FMA streaming kernel (1-2 rows per pass) beyond.
static cudaError_t launch_streaming(const GroupedProblem &p, cudaStream_t s)
{
    if (decode_fits(p.k))
        return launch_decode_gemm(p, p.P > 4 * (int64_t)p.E ? 8 : 4, s);
    return launch_stream_gemm(p, 2, s);
}

// Shared shape checks; returns FP4_OK or the status to report.
static int check_shape(int64_t rows, int64_t n, int64_t k)
{
    if (rows < 0 || n < 0 || k < 0)
        return FP4_ERR_ARG;
    if (k == 0 || (k % 128) != 0 || n == 0)
        return FP4_ERR_SHAPE;
    if (k > (1 << 20) || n > (1 << 24) || rows > ((int64_t)1 << 31))
        return FP4_ERR_SHAPE;
    if (stream_max_rows_per_pass((int)k) == 0)
        return FP4_ERR_SHAPE;
    return FP4_OK;
}

static int run_grouped(GroupedProblem p, void *workspace, size_t ws_bytes, cudaStream_t s)
{
    p.err = device_error_word();
    if (!p.err)
        return record(cudaGetLastError() != cudaSuccess ? cudaGetLastError()
                                                          : cudaErrorInvalidDevice);
    const bool have_ws =
        workspace != nullptr && ws_bytes >= tc_path_workspace(p.T, p.P, p.k, p.recipe);
    const int path = choose_path_for(p, have_ws);
    if (path == FP4_PATH_TC) {
        if (!tc_supported(p.n, p.k, p.recipe, p.E))
            return FP4_ERR_SHAPE;
        if (!tc_path_supported(p.n, p.k, p.recipe, p.E, p.w))
            return FP4_ERR_ALIGN;
        if (!have_ws)
            return FP4_ERR_WORKSPACE;
        if (p.codes_out) {  // the codes are not a by-product of the quantise pass: one act_quant
            const int st = record(launch_act_quant(p.x, p.codes_out, p.scales_out, p.P, p.k, s));
            if (st != FP4_OK)
                return st;
        }
        const int st = record(tc_path_quantize(p, workspace, s));
        if (st != FP4_OK)
            return st;
        return record(tc_path_gemm(p, workspace, s));
    }
    return record(launch_streaming(p, s));
}

} // namespace fp4moe

using namespace fp4moe;

extern "C" {

int act_quant_fp8(const float *x, uint8_t *codes, float *scales, int64_t rows, int64_t k,
                  void *stream)
{
    if (rows < 0 || k < 0)
        return FP4_ERR_ARG;
    if (k == 0 || k % 128 != 0)
        return FP4_ERR_SHAPE;
    if (rows == 0)
        return FP4_OK;
    if (!x || !codes || !scales)
        return FP4_ERR_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales))
        return FP4_ERR_ALIGN;
    return record(launch_act_quant(x, codes, scales, rows, k, (cudaStream_t)stream));
}

int fp4_gemm_mirror(const uint8_t *codes, const float *scales, const uint8_t *w,
                    const uint8_t *wscale, float scale2, int recipe, float *out, int64_t g,
                    int64_t n, int64_t k, void *stream)
{
    if (!recipe_ok(recipe))
        return FP4_ERR_ARG;
    int st = check_shape(g, n, k);
    if (st != FP4_OK)
        return st;
    if (n > 0x7FFFFFFF)
        return FP4_ERR_SHAPE;
    if (g == 0)
        return FP4_OK;
    if (!codes || !scales || !w || !wscale || !out)
        return FP4_ERR_ARG;
    return record(launch_mirror_gemm(codes, scales, w, wscale, scale2, recipe, out, g, n, k,
                                     (cudaStream_t)stream));
}

int fp4_swiglu_quant(const float *gate, const float *up, int64_t ld, float limit, int64_t rows,
                     int64_t inter, float *h_out, uint8_t *codes, float *scales, void *stream)
{
    if (rows < 0 || inter < 0 || !(limit > 0.0f) || !(limit < 3.0e38f))
        return FP4_ERR_ARG;
    if (inter == 0 || inter % 128 != 0 || ld < inter || ld % 4 != 0)
        return FP4_ERR_SHAPE;
    if (rows == 0)
        return FP4_OK;
    if (!gate || !up || !codes || !scales)
        return FP4_ERR_ARG;
    if (!aligned16(gate) || !aligned16(up) || !aligned16(codes) || !aligned16(scales) ||
        (h_out && !aligned16(h_out)))
        return FP4_ERR_ALIGN;
    return record(launch_swiglu_quant(gate, up, ld, limit, rows, inter, h_out, codes, scales,
                                      (cudaStream_t)stream));
}

int fp4_expert_gemm(const float *x, const uint8_t *w, const uint8_t *wscale, float scale2,
                    int recipe, float *out, int64_t g, int64_t n, int64_t k, uint8_t *codes_out,
                    float *scales_out, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!recipe_ok(recipe))
        return FP4_ERR_ARG;
    int st = check_shape(g, n, k);
    if (st != FP4_OK)
        return st;
    if (g == 0)
        return FP4_OK;
    if (!x || !w || !wscale || !out || ((codes_out == nullptr) != (scales_out == nullptr)))
        return FP4_ERR_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(wscale) || !aligned16(out) ||
        (codes_out && (!aligned16(codes_out) || !aligned16(scales_out))))
        return FP4_ERR_ALIGN;
    GroupedProblem p{};
    p.x = x;
    p.T = g;
    p.row_ids = nullptr;
    p.offsets = nullptr;
    p.E = 1;
    p.P = g;
    p.w = w;
    p.sc = wscale;
    p.scale2 = nullptr;
    p.scale2_host = scale2;
    p.recipe = recipe;
    p.out = out;
    p.n = (int)n;
    p.k = (int)k;
    p.codes_out = codes_out;
    p.scales_out = scales_out;
    return run_grouped(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

size_t fp4_grouped_workspace_size(int64_t num_tokens, int64_t total_rows, int64_t n, int64_t k,
                                  int recipe)
{
    if (num_tokens < 0 || !recipe_ok(recipe) || check_shape(total_rows, n, k) != FP4_OK)
        return 0;
    if (!tc_supported(n, k, recipe, 1))
        return 0;  // the shape always takes the streaming path, which needs no workspace
    return tc_path_workspace(num_tokens, total_rows, k, recipe);
}

int fp4_grouped_expert_gemm(const float *x, int64_t num_tokens, const int32_t *row_ids,
                            const int32_t *offsets, int num_experts, int64_t total_rows,
                            const uint8_t *w, const uint8_t *wscale, const float *scale2,
                            int recipe, float *out, int64_t n, int64_t k, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    if (!recipe_ok(recipe) || num_experts < 1 || num_experts > 65535 || num_tokens < 0)
        return FP4_ERR_ARG;
    int st = check_shape(total_rows, n, k);
    if (st != FP4_OK)
        return st;
    if (total_rows == 0)
        return FP4_OK;
    if (!x || !offsets || !w || !wscale || !out || (recipe == FP4_NVFP4 && !scale2))
        return FP4_ERR_ARG;
    if (!row_ids && num_tokens < total_rows)
        return FP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(w) || !aligned16(wscale) || !aligned16(out))
        return FP4_ERR_ALIGN;
    GroupedProblem p{};
    p.x = x;
    p.T = num_tokens;
    p.row_ids = row_ids;
    p.offsets = offsets;
    p.E = num_experts;
    p.P = total_rows;
    p.w = w;
    p.sc = wscale;
    p.scale2 = recipe == FP4_NVFP4 ? scale2 : nullptr;
    p.scale2_host = 1.0f;
    p.recipe = recipe;
    p.out = out;
    p.n = (int)n;
    p.k = (int)k;
    p.codes_out = nullptr;
    p.scales_out = nullptr;
    return run_grouped(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

// Shared checks of the two halves of the tensor-core path.
static int check_tc_call(int recipe, int64_t num_tokens, const int32_t *row_ids,
                         int64_t total_rows, int64_t n, int64_t k, const void *ws, size_t ws_bytes)
{
    if (!recipe_ok(recipe) || num_tokens < 0)
        return FP4_ERR_ARG;
    const int st = check_shape(total_rows, n, k);
    if (st != FP4_OK)
        return st;
    if (!tc_supported(n, k, recipe, 1))
        return FP4_ERR_SHAPE;
    if (!row_ids && num_tokens < total_rows)
        return FP4_ERR_SHAPE;
    if (total_rows > 0 &&
        (!ws || ws_bytes < tc_path_workspace(num_tokens, total_rows, k, recipe)))
        return FP4_ERR_WORKSPACE;
    return FP4_OK;
}

int fp4_grouped_quantize(const float *x, int64_t num_tokens, const int32_t *row_ids,
                         int64_t total_rows, int64_t k, int recipe, void *workspace,
                         size_t workspace_bytes, void *stream)
{
    int st = check_tc_call(recipe, num_tokens, row_ids, total_rows, 128, k, workspace,
                           workspace_bytes);
    if (st != FP4_OK)
        return st;
    if (total_rows == 0)
        return FP4_OK;
    if (!x)
        return FP4_ERR_ARG;
    if (!aligned16(x))
        return FP4_ERR_ALIGN;
    GroupedProblem p{};
    p.x = x;
    p.T = num_tokens;
    p.row_ids = row_ids;
    p.E = 1;
    p.P = total_rows;
    p.recipe = recipe;
    p.n = 128;
    p.k = (int)k;
    p.err = device_error_word();
    if (!p.err)
        return record(cudaErrorInvalidDevice);
    return record(tc_path_quantize(p, workspace, (cudaStream_t)stream));
}

int fp4_grouped_gemm_quantized(const void *workspace, size_t workspace_bytes,
                               int64_t num_tokens, const int32_t *row_ids,
                               const int32_t *offsets, int num_experts, int64_t total_rows,
                               const uint8_t *w, const uint8_t *wscale, const float *scale2,
                               int recipe, float *out, int64_t n, int64_t k, void *stream)
{
    if (num_experts < 1 || num_experts > 65535)
        return FP4_ERR_ARG;
    int st = check_tc_call(recipe, num_tokens, row_ids, total_rows, n, k, workspace,
                           workspace_bytes);
    if (st != FP4_OK)
        return st;
    if (!tc_supported(n, k, recipe, num_experts))
        return FP4_ERR_SHAPE;
    if (total_rows == 0)
        return FP4_OK;
    if (!offsets || !w || !wscale || !out || (recipe == FP4_NVFP4 && !scale2))
        return FP4_ERR_ARG;
    if (!aligned16(w) || !aligned16(wscale) || !aligned16(out) ||
        !tc_path_supported(n, k, recipe, num_experts, w))
        return FP4_ERR_ALIGN;
    GroupedProblem p{};
    p.T = num_tokens;
    p.row_ids = row_ids;
    p.offsets = offsets;
    p.E = num_experts;
    p.P = total_rows;
    p.w = w;
    p.sc = wscale;
    p.scale2 = recipe == FP4_NVFP4 ? scale2 : nullptr;
    p.scale2_host = 1.0f;
    p.recipe = recipe;
    p.out = out;
    p.n = (int)n;
    p.k = (int)k;
    p.err = device_error_word();
    if (!p.err)
        return record(cudaErrorInvalidDevice);
    return record(tc_path_gemm(p, workspace, (cudaStream_t)stream));
}

int fp4_grouped_gate_up_swiglu(const float *x, int64_t num_tokens, const int32_t *row_ids,
                               const int32_t *offsets, int num_experts, int64_t total_rows,
                               const uint8_t *w, const uint8_t *wscale, const float *scale2,
                               int recipe, float swiglu_limit, float *h, int64_t inter,
                               int64_t k, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!recipe_ok(recipe) || num_experts < 1 || num_experts > 65535 || num_tokens < 0 ||
        !(swiglu_limit > 0.0f) || !(swiglu_limit <= 3.0e38f))
        return FP4_ERR_ARG;
    if (inter < 64 || inter % 64 != 0)
        return FP4_ERR_SHAPE;
    const int64_t n = 2 * inter;
    int st = check_tc_call(recipe, num_tokens, row_ids, total_rows, n, k, workspace,
                           workspace_bytes);
    if (st != FP4_OK)
        return st;
    if (!tc_supported(n, k, recipe, num_experts))
        return FP4_ERR_SHAPE;
    if (total_rows == 0)
        return FP4_OK;
    if (!x || !offsets || !w || !wscale || !h || (recipe == FP4_NVFP4 && !scale2))
        return FP4_ERR_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(wscale) || !aligned16(h) ||
        !tc_path_supported(n, k, recipe, num_experts, w))
        return FP4_ERR_ALIGN;
    GroupedProblem p{};
    p.x = x;
    p.T = num_tokens;
    p.row_ids = row_ids;
    p.offsets = offsets;
    p.E = num_experts;
    p.P = total_rows;
    p.w = w;
    p.sc = wscale;
    p.scale2 = recipe == FP4_NVFP4 ? scale2 : nullptr;
    p.scale2_host = 1.0f;
    p.recipe = recipe;
    p.out = nullptr;
    p.n = (int)n;
    p.k = (int)k;
    p.err = device_error_word();
    if (!p.err)
        return record(cudaErrorInvalidDevice);
    st = record(tc_path_quantize(p, workspace, (cudaStream_t)stream));
    if (st != FP4_OK)
        return st;
    const SwigluOut sw{h, inter, swiglu_limit};
    return record(tc_path_gemm(p, workspace, (cudaStream_t)stream, &sw));
}

int fp4_route_topk(const float *logits, int64_t num_tokens, int num_experts, int topk,
                   int renormalize, int32_t *ids, float *weights, void *stream)
{
    if (num_tokens < 0 || num_experts < 1 || topk < 1)
        return FP4_ERR_ARG;
    if (num_experts > 1024 || topk > 32 || topk > num_experts)
        return FP4_ERR_SHAPE;
    if (num_tokens == 0)
        return FP4_OK;
    if (!logits || !ids || !weights)
        return FP4_ERR_ARG;
    if (!aligned16(logits) || !aligned16(ids) || !aligned16(weights))
        return FP4_ERR_ALIGN;
    return record(launch_route_topk(logits, num_tokens, num_experts, topk, renormalize, ids,
                                    weights, (cudaStream_t)stream));
}

size_t fp4_route_csr_workspace_size(int64_t num_tokens, int num_experts)
{
    if (num_tokens < 0 || num_experts < 1)
        return 0;
    return route_csr_workspace_bytes(num_tokens, num_experts);
}

int fp4_route_csr(const int32_t *ids, int64_t num_tokens, int topk, int num_experts,
                  int32_t *offsets, int32_t *row_ids, int32_t *pair_rows, void *workspace,
                  size_t workspace_bytes, void *stream)
{
    if (num_tokens < 0 || topk < 1 || num_experts < 1 || num_experts > 65535)
        return FP4_ERR_ARG;
    if (num_tokens * (int64_t)topk > ((int64_t)1 << 31) - 1)
        return FP4_ERR_SHAPE;
    if (!offsets || !workspace || (num_tokens > 0 && (!ids || !row_ids)))
        return FP4_ERR_ARG;
    if (workspace_bytes < route_csr_workspace_bytes(num_tokens, num_experts))
        return FP4_ERR_WORKSPACE;
    if (!aligned16(workspace))
        return FP4_ERR_ALIGN;
    unsigned *err = device_error_word();
    if (!err)
        return record(cudaErrorInvalidDevice);
    return record(launch_route_csr(ids, num_tokens, topk, num_experts, offsets, row_ids,
                                   pair_rows, workspace, err, (cudaStream_t)stream));
}

int fp4_moe_combine(const float *out, int64_t total_rows, const int32_t *pair_rows,
                    const float *weights, int64_t num_tokens, int topk, int64_t n, float *y,
                    void *stream)
{
    if (total_rows < 0 || num_tokens < 0 || topk < 1 || n < 0)
        return FP4_ERR_ARG;
    if (n == 0 || n % 4 != 0 || topk > 1024)
        return FP4_ERR_SHAPE;
    if (num_tokens == 0)
        return FP4_OK;
    if (!out || !pair_rows || !weights || !y)
        return FP4_ERR_ARG;
    if (!aligned16(out) || !aligned16(y))
        return FP4_ERR_ALIGN;
    unsigned *err = device_error_word();
    if (!err)
        return record(cudaErrorInvalidDevice);
    return record(launch_moe_combine(out, pair_rows, weights, num_tokens, topk, n, total_rows, y,
                                     err, (cudaStream_t)stream));
}

// ------------------------------------------------------------------ W4A4 variant

int act_quant_w4a4(const float *x, uint8_t *codes, uint8_t *scales, float *rowscale, int64_t rows,
                   int64_t k, void *stream)
{
    if (rows < 0 || k < 0)
        return FP4_ERR_ARG;
    if (k == 0 || k % 16 != 0 || k > (1 << 20) || rows > ((int64_t)1 << 31))
        return FP4_ERR_SHAPE;
    if (rows == 0)
        return FP4_OK;
    if (!x || !codes || !scales || !rowscale)
        return FP4_ERR_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(rowscale))
        return FP4_ERR_ALIGN;
    unsigned *err = device_error_word();
    if (!err)
        return record(cudaErrorInvalidDevice);
    return record(launch_act_quant_w4a4(x, nullptr, rows, rows, k, codes, scales, rowscale, err,
                                        (cudaStream_t)stream));
}

// Shape checks of the W4A4 calls (k a multiple of 256: the GEMM's stage).
static int check_w4a4_shape(int64_t num_tokens, bool have_row_ids, int64_t total_rows,
                            int64_t n, int64_t k)
{
    if (num_tokens < 0 || total_rows < 0 || n < 0 || k < 0)
        return FP4_ERR_ARG;
    if (k < 256 || k % 256 != 0 || n == 0 || k > (1 << 20) || n > (1 << 24) ||
        total_rows > ((int64_t)1 << 31))
        return FP4_ERR_SHAPE;
    if (!have_row_ids && num_tokens < total_rows)
        return FP4_ERR_SHAPE;
    return FP4_OK;
}

size_t fp4_w4a4_workspace_size(int64_t num_tokens, int64_t total_rows, int64_t k)
{
    if (check_w4a4_shape(num_tokens, true, total_rows, 1, k) != FP4_OK)
        return 0;
    return w4a4_workspace_bytes(num_tokens, total_rows, k);
}

int fp4_w4a4_quantize(const float *x, int64_t num_tokens, const int32_t *row_ids,
                      int64_t total_rows, int64_t k, void *workspace, size_t workspace_bytes,
                      void *stream)
{
    int st = check_w4a4_shape(num_tokens, row_ids != nullptr, total_rows, 1, k);
    if (st != FP4_OK)
        return st;
    if (total_rows == 0)
        return FP4_OK;
    if (!x)
        return FP4_ERR_ARG;
    if (!workspace || workspace_bytes < w4a4_workspace_bytes(num_tokens, total_rows, k))
        return FP4_ERR_WORKSPACE;
    if (!aligned16(x))
        return FP4_ERR_ALIGN;
    GroupedProblem p{};
    p.x = x;
    p.T = num_tokens;
    p.row_ids = row_ids;
    p.E = 1;
    p.P = total_rows;
    p.recipe = FP4_NVFP4;
    p.n = 1;
    p.k = (int)k;
    p.err = device_error_word();
    if (!p.err)
        return record(cudaErrorInvalidDevice);
    return record(launch_w4a4_quantize(p, workspace, (cudaStream_t)stream));
}

int fp4_w4a4_gemm_quantized(const void *workspace, size_t workspace_bytes, int64_t num_tokens,
                            const int32_t *row_ids, const int32_t *offsets, int num_experts,
                            int64_t total_rows, const uint8_t *w, const uint8_t *wscale,
                            const float *scale2, float *out, int64_t n, int64_t k, void *stream)
{
    if (num_experts < 1 || num_experts > 65535)
        return FP4_ERR_ARG;
    int st = check_w4a4_shape(num_tokens, row_ids != nullptr, total_rows, n, k);
    if (st != FP4_OK)
        return st;
    if (!w4a4_supported(n, k, num_experts))
        return FP4_ERR_SHAPE;
    if (total_rows == 0)
        return FP4_OK;
    if (!offsets || !w || !wscale || !scale2 || !out)
        return FP4_ERR_ARG;
    if (!workspace || workspace_bytes < w4a4_workspace_bytes(num_tokens, total_rows, k))
        return FP4_ERR_WORKSPACE;
    if (!aligned16(w) || !aligned16(wscale) || !aligned16(out))
        return FP4_ERR_ALIGN;
    GroupedProblem p{};
    p.T = num_tokens;
    p.row_ids = row_ids;
    p.offsets = offsets;
    p.E = num_experts;
    p.P = total_rows;
    p.w = w;
    p.sc = wscale;
    p.scale2 = scale2;
    p.recipe = FP4_NVFP4;
    p.out = out;
    p.n = (int)n;
    p.k = (int)k;
    p.err = device_error_word();
    if (!p.err)
        return record(cudaErrorInvalidDevice);
    return record(launch_w4a4_gemm(p, workspace, (cudaStream_t)stream));
}

int fp4_grouped_expert_gemm_w4a4(const float *x, int64_t num_tokens, const int32_t *row_ids,
                                 const int32_t *offsets, int num_experts, int64_t total_rows,
                                 const uint8_t *w, const uint8_t *wscale, const float *scale2,
                                 float *out, int64_t n, int64_t k, void *workspace,
                                 size_t workspace_bytes, void *stream)
{
    if (num_experts < 1 || num_experts > 65535)
        return FP4_ERR_ARG;
    int st = check_w4a4_shape(num_tokens, row_ids != nullptr, total_rows, n, k);
    if (st != FP4_OK)
        return st;
    if (!w4a4_supported(n, k, num_experts))
        return FP4_ERR_SHAPE;
    if (total_rows == 0)
        return FP4_OK;
    if (!x)
        return FP4_ERR_ARG;
    st = fp4_w4a4_quantize(x, num_tokens, row_ids, total_rows, k, workspace, workspace_bytes,
                           stream);
    if (st != FP4_OK)
        return st;
    return fp4_w4a4_gemm_quantized(workspace, workspace_bytes, num_tokens, row_ids, offsets,
                                   num_experts, total_rows, w, wscale, scale2, out, n, k, stream);
}

double fp4_w4a4_error_ops(int64_t k)
{
    // the k/16 model of the other tensor-core paths (one rounding per 16-group of the f32
    // accumulation) plus the two epilogue multiplies (r, scale2) and one
    return (double)(k / 16) + 3.0;
}

int fp4_gemm_path(int64_t total_rows, int num_experts, int64_t n, int64_t k, int recipe,
                  int have_workspace)
{
    return choose_path(total_rows, num_experts, n, k, recipe, have_workspace != 0);
}

double fp4_error_ops(int path, int recipe, int64_t k)
{
    if (path == FP4_PATH_TC)
        return tc_error_ops(recipe, k);
    return decode_fits(k) ? decode_error_ops(recipe, k) : stream_error_ops(recipe, k);
}

void fp4_force_path(int path)
{
    g_forced_path = path == FP4_PATH_STREAM || path == FP4_PATH_TC ? path : FP4_PATH_AUTO;
}

void fp4_test_stall_next_gemm(int64_t wait_limit_cycles)
{
    const long long lo = 1000000LL;  // no wait of a healthy launch comes near this
    if (wait_limit_cycles <= 0) {
        g_stall_limit = 0;
        return;
    }
    g_stall_limit = wait_limit_cycles < lo ? lo
                    : wait_limit_cycles > kTimeoutCycles ? kTimeoutCycles
                                                         : (long long)wait_limit_cycles;
}

int fp4_get_device_error(void *stream, unsigned *bits)
{
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess)
        return record(e);
    unsigned v = 0u, zero = 0u;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess)
        return record(e);
    if (bits)
        *bits = v;
    return v ? FP4_ERR_DEVICE : FP4_OK;
}

const char *fp4_last_error(void)
{
    return g_last_error;
}

const char *fp4_status_string(int status)
{
    switch (status) {
    case FP4_OK: return "FP4_OK";
    case FP4_ERR_ARG: return "FP4_ERR_ARG";
    case FP4_ERR_SHAPE: return "FP4_ERR_SHAPE";
    case FP4_ERR_ALIGN: return "FP4_ERR_ALIGN";
    case FP4_ERR_LAUNCH: return "FP4_ERR_LAUNCH";
    case FP4_ERR_DEVICE: return "FP4_ERR_DEVICE";
    case FP4_ERR_WORKSPACE: return "FP4_ERR_WORKSPACE";
    default: return "FP4_ERR_UNKNOWN";
    }
}

} // extern "C"
