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
// k order inside a 64-k chunk. Lane (g, c) = (lane / 4, lane % 4) loads bytes 8c..8c+7
// of weight rows g and g+8, i.e. physical k 16c..16c+15 (one NVFP4 scale group). The
// MMA's k index is a relabelling of physical k, applied identically to A and B (the terms
// of a dot product can be taken in any order): in MMA step s (0..3) of the chunk,
// fragment k {2c, 2c+1} is physical k 16c + 4s + {0, 1} and fragment k {2c+8, 2c+9} is
// 16c + 4s + {2, 3}. A lane's A registers are then bytes 2s and 2s+1 of its own loads,
// and its B registers one 8-byte shared-memory read of activation row g.
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
constexpr int kDecRowPad = 4;  // f16 elements after each activation row: conflict-free B reads
constexpr int kDecU = 4;       // 64-k chunks whose loads are issued together

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

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
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
// shared memory, row stride k + kDecRowPad. Rows >= `rows` are not written: lanes whose
// B row is past the pass use zero registers instead.
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
        *reinterpret_cast<uint2 *>(act + (size_t)r * ld + g * 128 + lane * 4) = h;
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

// The scale bytes lane c needs for chunks ch0 .. ch0+kDecU-1 of one weight row, byte u =
// chunk ch0+u (NVFP4: group 4ch + c; MXFP4: group 2ch + c/2).
// The packing below takes exactly four chunks: 16 NVFP4 (8 MXFP4) scale bytes, one
// aligned vector load.
static_assert(kDecU == 4, "load_scales packs four chunks' scale bytes");

template <int GS>
__device__ __forceinline__ uint32_t load_scales(const uint8_t *srow, int ch0, int nch, int c,
                                                bool vec)
{
    if (vec && ch0 + kDecU <= nch) {
        if (GS == 16) {
            const uint4 v = *reinterpret_cast<const uint4 *>(srow + ch0 * 4);
            const uint32_t sel = (uint32_t)c;
            uint32_t lo, hi;
            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(v.x), "r"(v.y), "r"(sel | ((sel + 4) << 4)));
            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(v.z), "r"(v.w), "r"(sel | ((sel + 4) << 4)));
            uint32_t r;
            asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(r) : "r"(lo), "r"(hi));
            return r;
        } else {
            const uint2 v = *reinterpret_cast<const uint2 *>(srow + ch0 * 2);
            const uint32_t b = (uint32_t)(c >> 1);
            uint32_t r;
            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r)
                : "r"(v.x), "r"(v.y), "r"(b | ((b + 2) << 4) | ((b + 4) << 8) | ((b + 6) << 12)));
            return r;
        }
    }
    uint32_t r = 0;
#pragma unroll
    for (int u = 0; u < kDecU; ++u)
        if (ch0 + u < nch)
            r |= (uint32_t)srow[GS == 16 ? (ch0 + u) * 4 + c : (ch0 + u) * 2 + (c >> 1)] << (8 * u);
    return r;
}

// FULL: k is a multiple of 256, so every batch has four chunks and the scale rows are
// 16-byte aligned; no per-chunk checks.
template <int GS, bool F16, bool FULL, int PR>
__device__ __forceinline__ void decode_pass(const GroupedProblem &p, const uint16_t *act,
                                            const float *rowscale, const int *rowok, int64_t c0,
                                            int rows, const uint8_t *wexp, const uint8_t *sexp,
                                            float s2)
{
    const int k = p.k, n = p.n, ld = k + kDecRowPad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int colA = blockIdx.x * kDecCols + warp * kDecRowsPerWarp + g, colB = colA + 8;
    // Rows past n read row n-1 and B columns past the pass read the last row the buffer
    // holds: the loads need no predicate, and those outputs are never stored (an output
    // depends only on its own A row and B column).
    const int rA = min(colA, n - 1), rB = min(colB, n - 1);
    const uint8_t *wA = wexp + (size_t)rA * (k / 2) + c * 8;
    const uint8_t *wB = wexp + (size_t)rB * (k / 2) + c * 8;
    const uint8_t *sA = sexp + (size_t)rA * (k / GS);
    const uint8_t *sB = sexp + (size_t)rB * (k / GS);
    const uint16_t *bro = act + (size_t)min(g, PR - 1) * ld + 16 * c;  // activation row n = g
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int nch = k / 64;
    for (int ch0 = 0; ch0 < nch; ch0 += kDecU) {
        uint2 wa[kDecU], wb[kDecU];
#pragma unroll
        for (int u = 0; u < kDecU; ++u) {
            const bool in = FULL || ch0 + u < nch;
            wa[u] = in ? __ldcs(reinterpret_cast<const uint2 *>(wA + (ch0 + u) * 32))
                       : make_uint2(0u, 0u);
            wb[u] = in ? __ldcs(reinterpret_cast<const uint2 *>(wB + (ch0 + u) * 32))
                       : make_uint2(0u, 0u);
        }
        const uint32_t sa = load_scales<GS>(sA, ch0, nch, c, FULL);
        const uint32_t sb = load_scales<GS>(sB, ch0, nch, c, FULL);
        // NVFP4 f16 route: the four chunks' scales as f16, two per word
        uint32_t sA01 = 0, sA23 = 0, sB01 = 0, sB23 = 0;
        if (F16) {
            sA01 = e4m3x2_to_f16x2(sa & 0xFFFFu);
            sA23 = e4m3x2_to_f16x2(sa >> 16);
            sB01 = e4m3x2_to_f16x2(sb & 0xFFFFu);
            sB23 = e4m3x2_to_f16x2(sb >> 16);
        }
#pragma unroll
        for (int u = 0; u < kDecU; ++u) {
            const int ch = ch0 + u;
            if (!FULL && ch >= nch)
                break;
            uint32_t hA[8], hB[8];
            e2m1x8_to_f16x8(wa[u].x, *reinterpret_cast<uint32_t(*)[4]>(&hA[0]));
            e2m1x8_to_f16x8(wa[u].y, *reinterpret_cast<uint32_t(*)[4]>(&hA[4]));
            e2m1x8_to_f16x8(wb[u].x, *reinterpret_cast<uint32_t(*)[4]>(&hB[0]));
            e2m1x8_to_f16x8(wb[u].y, *reinterpret_cast<uint32_t(*)[4]>(&hB[4]));
            if (F16) {
                const uint32_t wA2 = (u < 2) ? sA01 : sA23, wB2 = (u < 2) ? sB01 : sB23;
                const __half2 hA2 = *reinterpret_cast<const __half2 *>(&wA2);
                const __half2 hB2 = *reinterpret_cast<const __half2 *>(&wB2);
                const __half2 scA = (u & 1) ? __high2half2(hA2) : __low2half2(hA2);
                const __half2 scB = (u & 1) ? __high2half2(hB2) : __low2half2(hB2);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    __half2 a2 = *reinterpret_cast<__half2 *>(&hA[j]);
                    __half2 b2 = *reinterpret_cast<__half2 *>(&hB[j]);
                    a2 = __hmul2(a2, scA);
                    b2 = __hmul2(b2, scB);
                    hA[j] = *reinterpret_cast<uint32_t *>(&a2);
                    hB[j] = *reinterpret_cast<uint32_t *>(&b2);
                }
            } else {
                const uint32_t ba = (sa >> (8 * u)) & 0xFFu, bb = (sb >> (8 * u)) & 0xFFu;
                const float fA = (GS == 16) ? e4m3_to_f32(ba) : e8m0_to_f32(ba);
                const float fB = (GS == 16) ? e4m3_to_f32(bb) : e8m0_to_f32(bb);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    hA[j] = f16x2_scaled_bf16(hA[j], fA);
                    hB[j] = f16x2_scaled_bf16(hB[j], fB);
                }
            }
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t a[4] = {hA[2 * s], hB[2 * s], hA[2 * s + 1], hB[2 * s + 1]};
                const uint2 bv = *reinterpret_cast<const uint2 *>(bro + ch * 64 + 4 * s);
                if (F16)
                    mma_f16_16816(d, a, bv.x, bv.y);
                else
                    mma_bf16_16816(d, a, bv.x, bv.y);
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
