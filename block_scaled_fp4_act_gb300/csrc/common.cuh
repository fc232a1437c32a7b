// common.cuh -- device helpers shared by the library's kernels (sm_103a).
//
// Formats (memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs):
//   activation code : e4m3fn byte, per-128 power-of-two f32 scale (fn quant_rows)
//   weight          : E2M1 nibble pairs, low nibble = even k (struct ExpertRaw, mirror_gemm)
//   NVFP4 scale     : e4m3 byte per 16 weights, times the f32 scale2 of the tensor
//   MXFP4 scale     : e8m0 byte per 32 weights, 2^(e-127)
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace fp4moe {

// Sets FP4_DEVERR_* bits in the per-device error word whose address the host passes in.
__device__ __forceinline__ void raise_device_error(unsigned *err, unsigned bits)
{
    atomicOr(err, bits);
}

// ---------------------------------------------------------------- activation quantisation

// f32(1/448) as fn quant_rows forms it: (1.0f64 / 448.0) rounded to f32.
constexpr float kInv448 = (float)(1.0 / 448.0);

// Smallest power of two >= t for a finite normal t > 0 (t = amax * f32(1/448) with
// amax >= 1e-4 is always normal): keep t if its mantissa is zero, else round the
// exponent up.
__device__ __forceinline__ float pow2_ceil_normal(float t)
{
    const uint32_t b = __float_as_uint(t);
    if ((b & 0x007FFFFFu) == 0u)
        return t;
    return __uint_as_float((b & 0x7F800000u) + 0x00800000u);
}

// 1/s for a power of two s in [2^-126, 2^126]: exact, by exponent arithmetic.
__device__ __forceinline__ float pow2_reciprocal(float s)
{
    return __uint_as_float((254u << 23) - __float_as_uint(s));
}

// Group scale from the group's max |x| (fn quant_rows: floor 1e-4, times f32(1/448),
// pow2_ceil).
__device__ __forceinline__ float group_scale(float amax)
{
    amax = fmaxf(amax, 1e-4f);
    return pow2_ceil_normal(amax * kInv448);
}

// x/s clamped to +-448, as fn quant_rows does before encoding. x * (1/s) equals x / s
// bit for bit: both are the correctly rounded value of the same exact quotient.
__device__ __forceinline__ float scaled_clamped(float x, float inv_s)
{
    return fminf(fmaxf(x * inv_s, -448.0f), 448.0f);
}

// Two f32 -> two e4m3 bytes, round to nearest even, saturating to finite (inputs are
// already within +-448, so saturation never triggers). Low byte = `lo`.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// Four f32 -> four e4m3 bytes packed little-endian.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

// Two e4m3 bytes (low 16 bits) -> f16x2, exact (low byte -> low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes)
{
    uint32_t r;
    uint16_t v = (uint16_t)two_bytes;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

// ---------------------------------------------------------------- weight decoding

// One byte of two E2M1 nibbles -> f16x2 (low nibble = even k -> low half), exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low_bits)
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(r)
        : "r"(byte_in_low_bits));
    return r;
}

// Four bytes (eight nibbles) -> four f16x2 words, k order preserved.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// e4m3 byte -> f32 (exact): through f16.
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte)
{
    const uint32_t h2 = e4m3x2_to_f16x2(byte & 0xFFu);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// e8m0 byte -> f32: 2^(e-127); e = 0 is the subnormal 2^-127 (exact).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e)
{
    return e == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// acc + w.lo*a.lo, then + w.hi*a.hi: f16 operands, exact products, f32 adds (one
// rounding each). Keeps the k order of the pair.
__device__ __forceinline__ float fma2_f16_f32(uint32_t w2, uint32_t a2, float acc)
{
    float r;
    asm("{\n\t.reg .b16 wl, wh, al, ah;\n\t"
        "mov.b32 {wl, wh}, %1;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.f16 %0, wl, al, %3;\n\t"
        "fma.rn.f32.f16 %0, wh, ah, %0;\n\t}"
        : "=f"(r)
        : "r"(w2), "r"(a2), "f"(acc));
    return r;
}

// ---------------------------------------------------------------- memory

// 128-bit streaming load of read-once data (weights): no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// SwiGLU of one element with the swiglu_limit clamps (memra-engine 0.98.0,
// src/bin/dsv4_native_gemm_gate.rs, swiglu_limit saturation cell): up clamped on both
// sides, gate from above, both before the sigmoid, in f32 in the page's order. Shared by
// the standalone SwiGLU kernel and the fused gate/up epilogues, so both give the same bits.
__device__ __forceinline__ float swiglu_one(float gate, float up, float limit)
{
    const float u = fminf(fmaxf(up, -limit), limit);
    const float g = fminf(gate, limit);
    return g * (1.0f / (1.0f + expf(-g))) * u;
}

// ---------------------------------------------------------------- mbarriers

// Every pipeline wait is bounded by about a second of clock64 cycles.
constexpr long long kTimeoutCycles = 2000000000LL;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware (up to ~10 ms) until the phase
// completes instead of returning at once, so waiting warps do not take issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(10000000u)
                 : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `limit` clock64 cycles, setting the abort flag and the
// TIMEOUT bit. Returns false if this CTA is aborting (flag set here or elsewhere).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned *err, long long limit = kTimeoutCycles)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            raise_device_error(err, FP4_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used to drain in-flight work on abort).
// Returns false if the phase did not complete in time.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kTimeoutCycles / 4)
            return false;
    return true;
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Prefetch [addr, addr + bytes) into L2 (addr 16-byte aligned, bytes a multiple of 16), in
// pieces of at most 16 KB.
__device__ __forceinline__ void prefetch_l2(const void *addr, uint32_t bytes)
{
    const char *a = static_cast<const char *>(addr);
    for (uint32_t off = 0; off < bytes; off += 16384u) {
        const uint32_t n = bytes - off < 16384u ? bytes - off : 16384u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a + off), "r"(n) : "memory");
    }
}

// An L2 cache policy that evicts the lines it fetches first (for data read once).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D TMA tile load as tma_load_2d, with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_evict_first(uint32_t dst, const CUtensorMap *map, int x,
                                                        int y, uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
                 : "memory");
}

// 2-D TMA tile load into shared memory, completing on an mbarrier (x: innermost).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

// Hardware named barriers, executed by whole converged warps.
__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void named_arrive(int id, int threads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

} // namespace fp4moe
