// mirror.cu -- the quantized expert GEMM in the page's own kernel order, bit for bit.
//
// memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs, fn mirror_gemm (the CPU mirror
// of the page's dsv4_fp4_gemm_kernel): per output, 128 partials; partial t takes weight
// groups t, t + 128, ...; a group's gs products e4m3(a) * E2M1(w) are summed in k order
// in f32, the sum is multiplied by f32(ws * as) and added to the partial; then a fixed
// halving tree (offsets 64, 32, ..., 1) combines the partials. Every multiply and add is
// a separately rounded f32 operation (__fmul_rn / __fadd_rn: no contraction to FMA), so
// the result equals the mirror exactly. An instrument for bit-identity with the pages,
// not a fast path: one 128-thread CTA per output.
#include "common.cuh"

namespace fp4moe {

constexpr int kMirrorThreads = 128;

__device__ __forceinline__ float e2m1_to_f32(uint32_t nib)
{
    const uint32_t h2 = e2m1x2_to_f16x2(nib & 0xFu);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

template <int GS>
__global__ void __launch_bounds__(kMirrorThreads) mirror_gemm_kernel(
    const uint8_t *__restrict__ codes, const float *__restrict__ scales,
    const uint8_t *__restrict__ w, const uint8_t *__restrict__ wscale, float scale2,
    float *__restrict__ out, int64_t g, int64_t n, int64_t k)
{
    __shared__ float part[kMirrorThreads];
    const int t = threadIdx.x;
    const int64_t col = blockIdx.x;
    const int64_t ngroups = k / GS, kq = k / 128;
    const uint8_t *wrow = w + col * (k / 2);
    const uint8_t *srow = wscale + col * ngroups;
    for (int64_t r = blockIdx.y; r < g; r += gridDim.y) {
        const uint8_t *arow = codes + r * k;
        const float *asrow = scales + r * kq;
        float acc = 0.0f;
        for (int64_t j = t; j < ngroups; j += kMirrorThreads) {
            const int64_t k0 = j * GS;
            float sub = 0.0f;
#pragma unroll
            for (int i = 0; i < GS; ++i) {
                const int64_t kk = k0 + i;
                const uint32_t byte = wrow[kk >> 1];
                const uint32_t nib = (kk & 1) ? (byte >> 4) : (byte & 0xFu);
                sub = __fadd_rn(sub, __fmul_rn(e4m3_to_f32(arow[kk]), e2m1_to_f32(nib)));
            }
            const float ws = (GS == 16) ? __fmul_rn(e4m3_to_f32(srow[j]), scale2)
                                        : e8m0_to_f32(srow[j]);
            const float scl = __fmul_rn(ws, asrow[k0 / 128]);
            acc = __fadd_rn(acc, __fmul_rn(sub, scl));
        }
        part[t] = acc;
#pragma unroll
        for (int off = kMirrorThreads >> 1; off > 0; off >>= 1) {
            __syncthreads();
            if (t < off)
                part[t] = __fadd_rn(part[t], part[t + off]);
        }
        __syncthreads();
        if (t == 0)
            out[r * n + col] = part[0];
        __syncthreads();  // part[] is rewritten by the next row
    }
}

cudaError_t launch_mirror_gemm(const uint8_t *codes, const float *scales, const uint8_t *w,
                               const uint8_t *wscale, float scale2, int recipe, float *out,
                               int64_t g, int64_t n, int64_t k, cudaStream_t s)
{
    if (g == 0)
        return cudaSuccess;
    dim3 grid((unsigned)n, (unsigned)(g < 65535 ? g : 65535));
    if (recipe == FP4_NVFP4)
        mirror_gemm_kernel<16><<<grid, kMirrorThreads, 0, s>>>(codes, scales, w, wscale, scale2,
                                                                out, g, n, k);
    else
        mirror_gemm_kernel<32><<<grid, kMirrorThreads, 0, s>>>(codes, scales, w, wscale, scale2,
                                                                out, g, n, k);
    return cudaGetLastError();
}

} // namespace fp4moe
