// act_quant.cu -- per-row, per-128 FP8-E4M3 activation quantisation
// (fn quant_rows of memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs).
//
// One warp per 128-element group: each lane loads one float4 (coalesced 512 B per
// warp), the group amax is a shuffle max (order-free, so bit-exact with any order),
// the scale is a power of two, and each lane writes its four codes as one 32-bit word.
// HBM-bound: 4 B read + 1 B written per element, plus 4 B of scale per 128.
#include "common.cuh"

namespace fp4moe {

__global__ void __launch_bounds__(256) act_quant_kernel(const float *__restrict__ x,
                                                        uint8_t *__restrict__ codes,
                                                        float *__restrict__ scales,
                                                        int64_t groups)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < groups;
         g += warps) {
        const float4 v = __ldcs(reinterpret_cast<const float4 *>(x + g * 128) + lane);
        float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        amax = warp_max(amax);
        const float s = group_scale(amax);
        const float inv = pow2_reciprocal(s);
        const uint32_t q = e4m3x4(scaled_clamped(v.x, inv), scaled_clamped(v.y, inv),
                                  scaled_clamped(v.z, inv), scaled_clamped(v.w, inv));
        reinterpret_cast<uint32_t *>(codes + g * 128)[lane] = q;
        if (lane == 0)
            scales[g] = s;
    }
}

cudaError_t launch_act_quant(const float *x, uint8_t *codes, float *scales, int64_t rows,
                             int64_t k, cudaStream_t s)
{
    const int64_t groups = rows * (k / 128);
    if (groups == 0)
        return cudaSuccess;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (groups + 7) / 8;
    const int64_t cap = (int64_t)sms * 8;  // 8 CTAs of 8 warps per SM, grid-stride beyond
    const int blocks = (int)(want < cap ? want : cap);
    act_quant_kernel<<<blocks, 256, 0, s>>>(x, codes, scales, groups);
    return cudaGetLastError();
}

} // namespace fp4moe
