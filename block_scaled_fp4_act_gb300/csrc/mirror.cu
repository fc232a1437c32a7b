// mirror.cu -- the quantized expert GEMM in the summation order of the page's own kernel,
// bit for bit (memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs: the order that
// fn mirror_gemm reproduces on the CPU for the dsv4_fp4_gemm_kernel).
//
// The order, as a specification: an output is a pairwise tree over 128 partial sums.
//   group term  G_j  = (the gs products e4m3(code) * E2M1(nibble) of weight group j, added
//                      one by one in k order, in f32) * f32(ws_j * s_a), s_a the scale of
//                      the activation block holding the group
//   partial     P_t  = the f32 running sum of G_t, G_{t+128}, G_{t+256}, ... in that order
//   result           = P_0 after the levels w = 64, 32, ..., 1, each replacing P_t by
//                      P_t + P_{t+w} for t < w
// Every operation is a separately rounded f32 multiply or add (__fmul_rn / __fadd_rn: no
// contraction to FMA).
//
// Here one warp computes one output: lane l keeps the partials P_l, P_{l+32}, P_{l+64} and
// P_{l+96} in registers; the levels 64 and 32 combine them inside the lane, the levels 16
// down to 1 are shuffles. An instrument for bit-identity with the pages, not a fast path.
#include "common.cuh"

namespace fp4moe {

constexpr int kMirrorWarps = 4;  // outputs (columns) per CTA

__device__ __forceinline__ float e2m1_value(uint32_t nibble)
{
    const uint32_t h2 = e2m1x2_to_f16x2(nibble & 0xFu);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// G_j of one output: activation codes/scales of its row, nibbles/scales of its column.
template <int GS>
__device__ __forceinline__ float group_term(const uint8_t *__restrict__ act, const float *__restrict__ act_scale,
                                            const uint8_t *__restrict__ nib, const uint8_t *__restrict__ wsc,
                                            float scale2, int64_t j)
{
    const int64_t first = j * GS;
    float dot = 0.0f;
#pragma unroll
    for (int i = 0; i < GS; i += 2) {
        const uint32_t pair = nib[(first + i) >> 1];  // k = first + i (low), first + i + 1 (high)
        dot = __fadd_rn(dot, __fmul_rn(e4m3_to_f32(act[first + i]), e2m1_value(pair)));
        dot = __fadd_rn(dot, __fmul_rn(e4m3_to_f32(act[first + i + 1]), e2m1_value(pair >> 4)));
    }
    const float wscale = GS == 16 ? __fmul_rn(e4m3_to_f32(wsc[j]), scale2) : e8m0_to_f32(wsc[j]);
    return __fmul_rn(dot, __fmul_rn(wscale, act_scale[first / 128]));
}

template <int GS>
__global__ void __launch_bounds__(32 * kMirrorWarps) mirror_gemm_kernel(
    const uint8_t *__restrict__ codes, const float *__restrict__ scales,
    const uint8_t *__restrict__ w, const uint8_t *__restrict__ wscale, float scale2,
    float *__restrict__ out, int64_t g, int64_t n, int64_t k)
{
    const int lane = threadIdx.x & 31;
    const int64_t col = (int64_t)blockIdx.x * kMirrorWarps + (threadIdx.x >> 5);
    if (col >= n)
        return;  // whole warp
    const int64_t groups = k / GS;
    const uint8_t *nib = w + col * (k / 2);
    const uint8_t *wsc = wscale + col * groups;
    for (int64_t row = blockIdx.y; row < g; row += gridDim.y) {
        const uint8_t *act = codes + row * k;
        const float *act_scale = scales + row * (k / 128);
        float part[4];  // P_{lane + 32 q}
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float acc = 0.0f;
            for (int64_t j = lane + 32 * q; j < groups; j += 128)
                acc = __fadd_rn(acc, group_term<GS>(act, act_scale, nib, wsc, scale2, j));
            part[q] = acc;
        }
        part[0] = __fadd_rn(part[0], part[2]);  // w = 64: P_l += P_{l+64}, P_{l+32} += P_{l+96}
        part[1] = __fadd_rn(part[1], part[3]);
        float v = __fadd_rn(part[0], part[1]);  // w = 32
#pragma unroll
        for (int wdt = 16; wdt > 0; wdt >>= 1)  // lanes l < wdt take P_l + P_{l+wdt}
            v = __fadd_rn(v, __shfl_down_sync(0xFFFFFFFFu, v, wdt));
        if (lane == 0)
            out[row * n + col] = v;
    }
}

cudaError_t launch_mirror_gemm(const uint8_t *codes, const float *scales, const uint8_t *w,
                               const uint8_t *wscale, float scale2, int recipe, float *out,
                               int64_t g, int64_t n, int64_t k, cudaStream_t s)
{
    if (g == 0)
        return cudaSuccess;
    dim3 grid((unsigned)((n + kMirrorWarps - 1) / kMirrorWarps), (unsigned)(g < 65535 ? g : 65535));
    if (recipe == FP4_NVFP4)
        mirror_gemm_kernel<16><<<grid, 32 * kMirrorWarps, 0, s>>>(codes, scales, w, wscale, scale2,
                                                                  out, g, n, k);
    else
        mirror_gemm_kernel<32><<<grid, 32 * kMirrorWarps, 0, s>>>(codes, scales, w, wscale, scale2,
                                                                  out, g, n, k);
    return cudaGetLastError();
}

} // namespace fp4moe
