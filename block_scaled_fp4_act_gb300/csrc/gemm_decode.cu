// gemm_decode.cu -- decode-sized grouped expert GEMM on warp-level tensor-core fragments.
//
// Arithmetic (memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs, fn f64_ref): every
// product e4m3(a) * s_a * E2M1(w) * ws is formed exactly and summed in f32, as on the
// tcgen05 path, here with mma.sync m16n8k16 (f32 accumulate). A warp owns 16 weight rows
// (the MMA's M); the routed rows of one pass (up to 8) are its N, so one MMA consumes 256
// weights however few rows an expert has, and the CUDA cores only unpack nibbles.
//   A (weights):     f16(E2M1 * e4m3 scale)            NVFP4, f16 route (exact)
//                    bf16(E2M1 * scale)                 otherwise (exact)
//   B (activations): f16(code * 2^(m - M_row))          f16 route: every 128-block of the
//                                                       pass's rows within 2^15 of its row's
//                                                       largest, so exact down to 2^-24
//                    bf16(code * 2^m)                   otherwise (MXFP4 always)
//   out = (D * 2^M_row) * scale2
//
// k order inside a 128-k block. Lane (g, c) = (lane / 4, lane % 4) loads bytes
// 16c..16c+15 of the block's 64 bytes of weight rows g and g+8 (one 16-byte load each,
// four lanes covering 64 contiguous bytes of a row), i.e. physical k 32c..32c+31: two
// NVFP4 scale groups, one MXFP4 group. The MMA's k index is a relabelling of physical k,
// applied identically to A and B (the terms of a dot product can be taken in any order):
// in MMA step s (0..7) of the block, fragment k {2c, 2c+1} is physical k 32c + 4s + {0, 1}
// and fragment k {2c+8, 2c+9} is 32c + 4s + {2, 3}. A lane's A registers are then bytes
// 2s and 2s+1 of its own loads, and its B registers one 8-byte shared-memory read of
// activation row g: the four elements at 32c + 4s, i.e. 4-element group q = 8c + s,
// which the activation buffer stores at group q ^ ((q >> 4) & 1) so that the reads of a
// half-warp fall in 32 distinct banks.
//
// Summation: one f32 accumulation per MMA (k/16 of them), then the row scale (exact) and
// scale2, the same depth as the tcgen05 path.
#include "common.cuh"

#include <cuda_bf16.h>

namespace fp4moe {

constexpr int kDecThreads = 256;
constexpr int kDecRowsPerWarp = 16;
constexpr int kDecCols = (kDecThreads / 32) * kDecRowsPerWarp;  // 128 weight rows per CTA
constexpr int kDecMaxScaleGap = 15;
constexpr int kDecRowPad = 8;  // f16 elements after each activation row: conflict-free B reads

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// f16x2 of two E2M1 values times an f32 scale -> bf16x2, exactly (<= 6 significant bits).
__device__ __forceinline__ uint32_t f16x2_scaled_bf16(uint32_t h, float s)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y * s), "f"(f.x * s));
    return r;
}

__device__ __forceinline__ int f32_biased_exponent(float s)
{
    return (int)((__float_as_uint(s) >> 23) & 0xFF);
}

// act_quant of the pass's rows (fn quant_rows of the page) into 16-bit MMA operands in
// shared memory, row stride k + kDecRowPad. Rows >= `rows` are not written: the MMA
// columns they feed are never stored.
__device__ __forceinline__ void decode_prologue(const GroupedProblem &p, int64_t c0, int rows,
                                                uint16_t *act, float *ascale, float *rowscale,
                                                int *rowok, int *route_f16, bool write_codes)
{
    const int k = p.k, kq = k >> 7, ld = k + kDecRowPad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0)
        *route_f16 = (p.recipe == FP4_NVFP4) ? 1 : 0;
    // phase 1: per 128-group scale and codes; f16(code) into act
    for (int gi = warp; gi < rows * kq; gi += kDecThreads / 32) {
        const int r = gi / kq, g = gi - r * kq;
        uint2 h = make_uint2(0u, 0u);
        float s = 0.0f;
        int ok = 0;
        const int64_t pr = c0 + r;
        const int64_t t = p.row_ids ? (int64_t)p.row_ids[pr] : pr;
        if (t >= 0 && t < p.T) {
            ok = 1;
            const float4 v =
                *reinterpret_cast<const float4 *>(p.x + t * (int64_t)k + g * 128 + lane * 4);
            float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
            amax = warp_max(amax);
            s = group_scale(amax);
            const float inv = pow2_reciprocal(s);
            const uint32_t q = e4m3x4(scaled_clamped(v.x, inv), scaled_clamped(v.y, inv),
                                      scaled_clamped(v.z, inv), scaled_clamped(v.w, inv));
            h.x = e4m3x2_to_f16x2(q & 0xFFFFu);
            h.y = e4m3x2_to_f16x2(q >> 16);
            if (write_codes) {
                reinterpret_cast<uint32_t *>(p.codes_out + pr * k + g * 128)[lane] = q;
                if (lane == 0)
                    p.scales_out[pr * kq + g] = s;
            }
        } else if (lane == 0 && g == 0) {
            raise_device_error(p.err, FP4_DEVERR_ROW_ID);
        }
        // 4-element group q of a 128-block is stored at q ^ ((q >> 4) & 1) (see decode_pass)
        *reinterpret_cast<uint2 *>(act + (size_t)r * ld + g * 128 + 4 * (lane ^ ((lane >> 4) & 1))) = h;
        if (lane == 0) {
            ascale[r * kq + g] = s;
            if (g == 0)
                rowok[r] = ok;
        }
    }
    __syncthreads();
    // phase 2: per row, the largest block exponent M, and whether every block is within 2^15
    if (warp < rows) {
        const int r = warp;
        int mx = 0, mn = 255;
        for (int g = lane; g < kq; g += 32) {
            const float s = ascale[r * kq + g];
            if (s > 0.0f) {
                const int ex = f32_biased_exponent(s);
                mx = max(mx, ex);
                mn = min(mn, ex);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
            mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
        }
        if (lane == 0) {
            rowscale[r] = mx > 0 ? __uint_as_float((uint32_t)mx << 23) : 1.0f;
            if (mx > 0 && mx - mn > kDecMaxScaleGap)
                atomicAnd(route_f16, 0);
        }
    }
    __syncthreads();
    // phase 3: rescale in place: f16(code * 2^(m - M)) or bf16(code * 2^m), both exact
    const bool f16 = *route_f16 != 0;
    const int half = k >> 1;
    for (int e2 = threadIdx.x; e2 < rows * half; e2 += kDecThreads) {
        const int r = e2 / half, kk = (e2 - r * half) * 2;
        uint32_t *pv = reinterpret_cast<uint32_t *>(act + (size_t)r * ld + kk);
        const float s = ascale[r * kq + (kk >> 7)];
        const uint32_t hv = *pv;
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hv));
        uint32_t o;
        if (f16) {
            const float m = s * pow2_reciprocal(rowscale[r]);  // 2^(m - M) >= 2^-15, exact
            const __half2 v = __floats2half2_rn(f.x * m, f.y * m);
            o = *reinterpret_cast<const uint32_t *>(&v);
        } else {
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(f.y * s), "f"(f.x * s));
        }
        *pv = o;
    }
    __syncthreads();
}

// The scale bytes of weight row `srow` lane c needs for k-batch b (256 k: blocks 2b and
// 2b+1), packed as byte pairs: NVFP4 groups 16b + 2c, +1 (bits 0-15) and 16b + 8 + 2c, +1
// (bits 16-31); MXFP4 group 8b + c (bits 0-7) and 8b + 4 + c (bits 8-15). h1: block 2b+1
// exists. FULL: k % 256 == 0, so the batch's scale bytes are one aligned vector.
template <int GS, bool FULL>
__device__ __forceinline__ uint32_t batch_scales(const uint8_t *srow, int b, int c, bool h1)
{
    uint32_t lo, hi;
    if (GS == 16) {
        uint2 v0, v1 = make_uint2(0u, 0u);
        if (FULL) {
            const uint4 v = *reinterpret_cast<const uint4 *>(srow + b * 16);
            v0 = make_uint2(v.x, v.y);
            v1 = make_uint2(v.z, v.w);
        } else {
            v0 = *reinterpret_cast<const uint2 *>(srow + b * 16);
            if (h1)
                v1 = *reinterpret_cast<const uint2 *>(srow + b * 16 + 8);
        }
        lo = (c >> 1) ? v0.y : v0.x;
        hi = (c >> 1) ? v1.y : v1.x;
        const uint32_t o = 2u * (uint32_t)(c & 1);
        uint32_t r;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r)
            : "r"(lo), "r"(hi), "r"(o | ((o + 1) << 4) | ((o + 4) << 8) | ((o + 5) << 12)));
        return r;
    } else {
        if (FULL) {
            const uint2 v = *reinterpret_cast<const uint2 *>(srow + b * 8);
            lo = v.x;
            hi = v.y;
        } else {
            lo = *reinterpret_cast<const uint32_t *>(srow + b * 8);
            hi = h1 ? *reinterpret_cast<const uint32_t *>(srow + b * 8 + 4) : 0u;
        }
        uint32_t r;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(c | ((c + 4) << 4)));
        return r & 0xFFFFu;
    }
}

// FULL: k is a multiple of 256, so every batch has both 128-k blocks; no per-block checks.
template <int GS, bool F16, bool FULL, int PR>
__device__ __forceinline__ void decode_pass(const GroupedProblem &p, const uint16_t *act,
                                            const float *rowscale, const int *rowok, int64_t c0,
                                            int rows, const uint8_t *wexp, const uint8_t *sexp,
                                            float s2)
{
    const int k = p.k, n = p.n, ld = k + kDecRowPad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3, swz = c >> 1;
    const int colA = blockIdx.x * kDecCols + warp * kDecRowsPerWarp + g, colB = colA + 8;
    // Rows past n read row n-1 and B columns past the pass read the last row the buffer
    // holds: the loads need no predicate, and those outputs are never stored (an output
    // depends only on its own A row and B column).
    const int rA = min(colA, n - 1), rB = min(colB, n - 1);
    const uint8_t *wA = wexp + (size_t)rA * (k / 2) + c * 16;
    const uint8_t *wB = wexp + (size_t)rB * (k / 2) + c * 16;
    const uint8_t *sA = sexp + (size_t)rA * (k / GS);
    const uint8_t *sB = sexp + (size_t)rB * (k / GS);
    // activation row n = g; step 2w + t reads group 8c + (2w + (t ^ swz)) of its block
    const uint16_t *bro = act + (size_t)min(g, PR - 1) * ld + 32 * c;
    const uint16_t *bro_t[2] = {bro + 4 * swz, bro + 4 * (swz ^ 1)};
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int nblk = k / 128, nb = (nblk + 1) / 2;
    for (int b = 0; b < nb; ++b) {
        const bool h1 = FULL || 2 * b + 1 < nblk;
        uint4 wa[2], wb[2];
        wa[0] = __ldcs(reinterpret_cast<const uint4 *>(wA + b * 128));
        wb[0] = __ldcs(reinterpret_cast<const uint4 *>(wB + b * 128));
        wa[1] = h1 ? __ldcs(reinterpret_cast<const uint4 *>(wA + b * 128 + 64)) : make_uint4(0, 0, 0, 0);
        wb[1] = h1 ? __ldcs(reinterpret_cast<const uint4 *>(wB + b * 128 + 64)) : make_uint4(0, 0, 0, 0);
        const uint32_t sa = batch_scales<GS, FULL>(sA, b, c, h1);
        const uint32_t sb = batch_scales<GS, FULL>(sB, b, c, h1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (!FULL && h == 1 && !h1)
                break;
            const int blk = 2 * b + h;
            const uint32_t va[4] = {wa[h].x, wa[h].y, wa[h].z, wa[h].w};
            const uint32_t vb[4] = {wb[h].x, wb[h].y, wb[h].z, wb[h].w};
            __half2 scA_lo, scA_hi, scB_lo, scB_hi;  // f16 route: groups 2c and 2c+1
            float fA_lo = 0.0f, fA_hi = 0.0f, fB_lo = 0.0f, fB_hi = 0.0f;
            if (F16) {
                const uint32_t pa = e4m3x2_to_f16x2((sa >> (16 * h)) & 0xFFFFu);
                const uint32_t pb = e4m3x2_to_f16x2((sb >> (16 * h)) & 0xFFFFu);
                const __half2 ha = *reinterpret_cast<const __half2 *>(&pa);
                const __half2 hb = *reinterpret_cast<const __half2 *>(&pb);
                scA_lo = __low2half2(ha);
                scA_hi = __high2half2(ha);
                scB_lo = __low2half2(hb);
                scB_hi = __high2half2(hb);
            } else if (GS == 16) {
                fA_lo = e4m3_to_f32((sa >> (16 * h)) & 0xFFu);
                fA_hi = e4m3_to_f32((sa >> (16 * h + 8)) & 0xFFu);
                fB_lo = e4m3_to_f32((sb >> (16 * h)) & 0xFFu);
                fB_hi = e4m3_to_f32((sb >> (16 * h + 8)) & 0xFFu);
            } else {
                fA_lo = fA_hi = e8m0_to_f32((sa >> (8 * h)) & 0xFFu);
                fB_lo = fB_hi = e8m0_to_f32((sb >> (8 * h)) & 0xFFu);
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t hA[4], hB[4];
                e2m1x8_to_f16x8(va[w], hA);
                e2m1x8_to_f16x8(vb[w], hB);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (F16) {
                        __half2 a2 = *reinterpret_cast<__half2 *>(&hA[j]);
                        __half2 b2 = *reinterpret_cast<__half2 *>(&hB[j]);
                        a2 = __hmul2(a2, w < 2 ? scA_lo : scA_hi);
                        b2 = __hmul2(b2, w < 2 ? scB_lo : scB_hi);
                        hA[j] = *reinterpret_cast<uint32_t *>(&a2);
                        hB[j] = *reinterpret_cast<uint32_t *>(&b2);
                    } else {
                        hA[j] = f16x2_scaled_bf16(hA[j], w < 2 ? fA_lo : fA_hi);
                        hB[j] = f16x2_scaled_bf16(hB[j], w < 2 ? fB_lo : fB_hi);
                    }
                }
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const uint32_t a[4] = {hA[2 * t], hB[2 * t], hA[2 * t + 1], hB[2 * t + 1]};
                    const uint2 bv = *reinterpret_cast<const uint2 *>(bro_t[t] + blk * 128 + 8 * w);
                    if (F16)
                        mma_f16_16816(d, a, bv.x, bv.y);
                    else
                        mma_bf16_16816(d, a, bv.x, bv.y);
                }
            }
        }
    }
    // D: (row g, n = 2c, 2c+1) in d0, d1; (row g+8, the same n) in d2, d3
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int nn = 2 * c + (j & 1);
        const int col = (j < 2) ? colA : colB;
        if (nn < rows && col < n && rowok[nn]) {
            const float rs = F16 ? rowscale[nn] : 1.0f;
            p.out[(c0 + nn) * (int64_t)n + col] = (d[j] * rs) * s2;
        }
    }
}

// PR: most routed rows one pass holds (the MMA's N is 8; 4 halves the shared memory).
template <int GS, int PR>
__global__ void __launch_bounds__(kDecThreads, 4) decode_mma_kernel(const GroupedProblem p)
{
    extern __shared__ __align__(16) uint8_t smem_dec[];
    const int k = p.k, n = p.n, kq = k >> 7;
    uint16_t *act = reinterpret_cast<uint16_t *>(smem_dec);
    float *ascale = reinterpret_cast<float *>(smem_dec + (size_t)PR * (k + kDecRowPad) * 2);
    float *rowscale = ascale + PR * kq;
    int *rowok = reinterpret_cast<int *>(rowscale + PR);
    int *route_f16 = rowok + PR;

    const int e = blockIdx.y;
    int64_t r0 = 0, r1 = p.P;
    if (p.offsets) {
        r0 = p.offsets[e];
        r1 = p.offsets[e + 1];
        const bool bad = r0 < 0 || r1 < r0 || r1 > p.P || (e == 0 && r0 != 0) ||
                         (e == p.E - 1 && r1 != p.P);
        if (bad) {
            if (threadIdx.x == 0 && blockIdx.x == 0)
                raise_device_error(p.err, FP4_DEVERR_OFFSETS);
            return;
        }
    }
    if (r0 >= r1)
        return;
    const float s2 = (GS == 16) ? (p.scale2 ? p.scale2[e] : p.scale2_host) : 1.0f;
    const uint8_t *wexp = p.w + (size_t)e * n * ((size_t)k / 2);
    const uint8_t *sexp = p.sc + (size_t)e * n * ((size_t)k / GS);
    const bool write_codes = p.codes_out != nullptr && blockIdx.x == 0;
    for (int64_t c0 = r0; c0 < r1; c0 += PR) {
        const int rows = (int)((r1 - c0) < PR ? (r1 - c0) : PR);
        decode_prologue(p, c0, rows, act, ascale, rowscale, rowok, route_f16, write_codes);
        const bool full = (k & 255) == 0;
        if (GS == 16 && *route_f16) {
            if (full)
                decode_pass<GS, true, true, PR>(p, act, rowscale, rowok, c0, rows, wexp, sexp, s2);
            else
                decode_pass<GS, true, false, PR>(p, act, rowscale, rowok, c0, rows, wexp, sexp, s2);
        } else {
            if (full)
                decode_pass<GS, false, true, PR>(p, act, rowscale, rowok, c0, rows, wexp, sexp, s2);
            else
                decode_pass<GS, false, false, PR>(p, act, rowscale, rowok, c0, rows, wexp, sexp, s2);
        }
        __syncthreads();  // act and the route flag are rewritten by the next pass
    }
}

static size_t decode_smem_bytes(int pr, int64_t k)
{
    return (size_t)pr * (k + kDecRowPad) * 2 + (size_t)pr * (k / 128) * 4 + (size_t)pr * 8 + 16;
}

constexpr size_t kDecSmemLimit = 227 * 1024;

bool decode_fits(int64_t k)
{
    return decode_smem_bytes(4, k) <= kDecSmemLimit;
}

template <int GS, int PR>
static cudaError_t launch_pr(const GroupedProblem &p, cudaStream_t s)
{
    const size_t smem = decode_smem_bytes(PR, p.k);
    auto kern = decode_mma_kernel<GS, PR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)((p.n + kDecCols - 1) / kDecCols), (unsigned)p.E);
    kern<<<grid, kDecThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode_gemm(const GroupedProblem &p, int rows_per_pass, cudaStream_t s)
{
    const bool nv = p.recipe == FP4_NVFP4;
    if (rows_per_pass <= 4 || decode_smem_bytes(8, p.k) > kDecSmemLimit)
        return nv ? launch_pr<16, 4>(p, s) : launch_pr<32, 4>(p, s);
    return nv ? launch_pr<16, 8>(p, s) : launch_pr<32, 8>(p, s);
}

// One f32 accumulation per k16 MMA step, the row-scale multiply (exact) and the scale2
// multiply; NVFP4 adds the f32 rounding of ws = e4m3 * scale2 that the f64 reference takes
// where this path multiplies by scale2 last, and that of the final product.
double decode_error_ops(int recipe, int64_t k)
{
    return (double)(k / 16) + (recipe == FP4_NVFP4 ? 2.0 : 0.0) + 1.0;
}

} // namespace fp4moe
