// swiglu.cu -- SwiGLU with the swiglu_limit clamps, fused with the per-128 FP8-E4M3
// requantisation of its output (the input of the down projection).
//
// The page (memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs, swiglu_limit
// saturation cell and the f64 check of main) computes, per element,
//   u = clamp(up, -L, L),  g = min(gate, L),  h = g * (1 / (1 + exp(-g))) * u
// (up clamped on both sides, gate on one side, both before the sigmoid), then quantises h
// with fn quant_rows before the down projection. One warp per 128-element group of a
// row: each lane loads a float4 of gate and of up, forms h in f32 in the page's order
// (expf: accurate to a few ulps, the class the page's check allows), and the group is
// quantised exactly as act_quant_kernel does, so the codes are act_quant of this h.
// HBM-bound: 8 B read + 1 B of code (+ 4 B of h if asked) per element, 4 B of scale per 128.
#include "common.cuh"

namespace fp4moe {

// h of one lane's four elements, then the group's scale and codes (act_quant_kernel's steps).
__device__ __forceinline__ void swiglu_group(const float4 gv, const float4 uv, float limit,
                                             int64_t gi, int64_t o, int lane,
                                             float *__restrict__ h_out,
                                             uint8_t *__restrict__ codes,
                                             float *__restrict__ scales)
{
    float4 h;
    h.x = swiglu_one(gv.x, uv.x, limit);
    h.y = swiglu_one(gv.y, uv.y, limit);
    h.z = swiglu_one(gv.z, uv.z, limit);
    h.w = swiglu_one(gv.w, uv.w, limit);
    if (h_out)
        *reinterpret_cast<float4 *>(h_out + o) = h;
    float amax = fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w)));
    amax = warp_max(amax);
    const float s = group_scale(amax);
    const float inv = pow2_reciprocal(s);
    const uint32_t q = e4m3x4(scaled_clamped(h.x, inv), scaled_clamped(h.y, inv),
                              scaled_clamped(h.z, inv), scaled_clamped(h.w, inv));
    reinterpret_cast<uint32_t *>(codes + o)[0] = q;
    if (lane == 0)
        scales[gi] = s;
}

// A warp takes two groups per iteration and issues all four 512-byte loads before
// computing, to keep more bytes in flight per SM.
__global__ void __launch_bounds__(256) swiglu_quant_kernel(
    const float *__restrict__ gate, const float *__restrict__ up, int64_t ld, float limit,
    int64_t inter, int64_t groups, float *__restrict__ h_out, uint8_t *__restrict__ codes,
    float *__restrict__ scales)
{
    const int lane = threadIdx.x & 31;
    const int64_t gpr = inter / 128;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t g0 = 2 * ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
         g0 < groups; g0 += 2 * warps) {
        const int64_t r0 = g0 / gpr, c0 = (g0 - r0 * gpr) * 128 + lane * 4;
        const bool two = g0 + 1 < groups;
        const int64_t g1 = two ? g0 + 1 : g0;
        const int64_t r1 = g1 / gpr, c1 = (g1 - r1 * gpr) * 128 + lane * 4;
        const float4 gv0 = __ldcs(reinterpret_cast<const float4 *>(gate + r0 * ld + c0));
        const float4 uv0 = __ldcs(reinterpret_cast<const float4 *>(up + r0 * ld + c0));
        const float4 gv1 = __ldcs(reinterpret_cast<const float4 *>(gate + r1 * ld + c1));
        const float4 uv1 = __ldcs(reinterpret_cast<const float4 *>(up + r1 * ld + c1));
        swiglu_group(gv0, uv0, limit, g0, r0 * inter + c0, lane, h_out, codes, scales);
        if (two)
            swiglu_group(gv1, uv1, limit, g1, r1 * inter + c1, lane, h_out, codes, scales);
    }
}

cudaError_t launch_swiglu_quant(const float *gate, const float *up, int64_t ld, float limit,
                                int64_t rows, int64_t inter, float *h_out, uint8_t *codes,
                                float *scales, cudaStream_t s)
{
    const int64_t groups = rows * (inter / 128);
    if (groups == 0)
        return cudaSuccess;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (groups + 15) / 16;  // two groups per warp, 8 warps per CTA
    const int64_t cap = (int64_t)sms * 8;     // 8 CTAs of 8 warps per SM, grid-stride beyond
    const int blocks = (int)(want < cap ? want : cap);
    swiglu_quant_kernel<<<blocks, 256, 0, s>>>(gate, up, ld, limit, inter, groups, h_out, codes,
                                               scales);
    return cudaGetLastError();
}

} // namespace fp4moe
