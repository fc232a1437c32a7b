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
//
// Two kernels share this MMA step (mma_block): decode_tma_kernel, whose weights arrive by
// TMA into a shared-memory ring (k a multiple of 512, at most 1024 experts, 16-byte aligned
// banks; its lanes read the same bytes from the ring), and decode_mma_kernel, whose lanes
// load their bytes from global memory themselves (every other shape).
#include "common.cuh"
#include "tma_host.h"

#include <cuda_bf16.h>

#include <algorithm>

namespace fp4moe {

constexpr int kDecThreads = 256;
constexpr int kDecRowsPerWarp = 16;
constexpr int kDecCols = (kDecThreads / 32) * kDecRowsPerWarp;  // 128 weight rows per CTA
constexpr int kDecMaxScaleGap = 15;
constexpr int kDecRowPad = 8;  // f16 elements after each activation row: conflict-free B reads
constexpr size_t kDecSmemLimit = 227 * 1024;

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

// Barrier of the NT threads that run the prologue and the MMAs (the whole CTA of
// decode_mma_kernel; the consumer warps of decode_tma_kernel, whose producer warp stays out).
template <int NT>
__device__ __forceinline__ void consumer_sync()
{
    named_sync(1, NT);
}

// act_quant of the pass's rows (fn quant_rows of the page) into 16-bit MMA operands in
// shared memory, row stride k + kDecRowPad, by the first NT threads of the CTA (at least
// 8 warps). Rows >= `rows` are not written: the MMA columns they feed are never stored.
// toks: the rows' token ids already in shared memory, or null (read through row_ids).
template <int NT>
__device__ __forceinline__ void decode_prologue(const GroupedProblem &p, int64_t c0, int rows,
                                                uint16_t *act, float *ascale, float *rowscale,
                                                int *rowok, int *route_f16, bool write_codes,
                                                const int32_t *toks = nullptr)
{
    const int k = p.k, kq = k >> 7, ld = k + kDecRowPad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0)
        *route_f16 = (p.recipe == FP4_NVFP4) ? 1 : 0;
    constexpr int NW = NT / 32, kBatch = 4;
    // phase 1: per 128-group scale and codes; f16(code) into act. A warp loads the
    // activations of kBatch groups before reducing any, so that they are in flight together.
    for (int gb = warp; gb < rows * kq; gb += NW * kBatch) {
        float4 v[kBatch];
        int64_t tt[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int gi = gb + b * NW;
            v[b] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            tt[b] = -1;
            if (gi < rows * kq) {
                const int r = gi / kq, g = gi - r * kq;
                const int64_t pr = c0 + r;
                const int64_t t = toks ? (int64_t)toks[r] : p.row_ids ? (int64_t)p.row_ids[pr] : pr;
                tt[b] = t;
                if (t >= 0 && t < p.T)
                    v[b] = *reinterpret_cast<const float4 *>(p.x + t * (int64_t)k + g * 128 + lane * 4);
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int gi = gb + b * NW;
            if (gi >= rows * kq)
                break;
            const int r = gi / kq, g = gi - r * kq;
            const int64_t pr = c0 + r;
            const int64_t t = tt[b];
            uint2 h = make_uint2(0u, 0u);
            float s = 0.0f;
            int ok = 0;
            if (t >= 0 && t < p.T) {
                ok = 1;
                float amax = fmaxf(fmaxf(fabsf(v[b].x), fabsf(v[b].y)),
                                   fmaxf(fabsf(v[b].z), fabsf(v[b].w)));
                amax = warp_max(amax);
                s = group_scale(amax);
                const float inv = pow2_reciprocal(s);
                const uint32_t q = e4m3x4(scaled_clamped(v[b].x, inv), scaled_clamped(v[b].y, inv),
                                          scaled_clamped(v[b].z, inv), scaled_clamped(v[b].w, inv));
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
    }
    consumer_sync<NT>();
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
    consumer_sync<NT>();
    // phase 3: rescale in place: f16(code * 2^(m - M)) or bf16(code * 2^m), both exact;
    // eight elements (16 bytes, inside one 128-block) per thread and step
    const bool f16 = *route_f16 != 0;
    const int tid = threadIdx.x % NT;
    for (int r = 0; r < rows; ++r) {
        const float rinv = f16 ? pow2_reciprocal(rowscale[r]) : 1.0f;
        for (int c = tid; c < (k >> 3); c += NT) {
            uint4 *pv = reinterpret_cast<uint4 *>(act + (size_t)r * ld + c * 8);
            const float s = ascale[r * kq + (c >> 4)];
            const float m = f16 ? s * rinv : s;  // f16: 2^(m - M) >= 2^-15, exact
            uint4 v = *pv;
            uint32_t *w = &v.x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[j]));
                if (f16) {
                    const __half2 h2 = __floats2half2_rn(f.x * m, f.y * m);
                    w[j] = *reinterpret_cast<const uint32_t *>(&h2);
                } else {
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[j]) : "f"(f.y * m), "f"(f.x * m));
                }
            }
            *pv = v;
        }
    }
    consumer_sync<NT>();
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

// One 128-k block of a warp's 16-row x 8-column MMA tile. wa, wb: the lane's 16 nibble
// bytes of its A-fragment rows g and g + 8 (physical k 32c..32c+31 of the block); sa, sb:
// their scale bytes for this block (NVFP4: two e4m3 bytes, groups 2c in bits 0-7 and
// 2c + 1 in bits 8-15; MXFP4: one e8m0 byte, group c); bro_t: the lane's activation row
// pointers (see decode_pass); blk: the block's index along k.
template <int GS, bool F16>
__device__ __forceinline__ void mma_block(float (&d)[4], const uint4 &wa, const uint4 &wb,
                                          uint32_t sa, uint32_t sb,
                                          const uint16_t *const (&bro_t)[2], int blk)
{
    const uint32_t va[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t vb[4] = {wb.x, wb.y, wb.z, wb.w};
    __half2 scA_lo, scA_hi, scB_lo, scB_hi;  // f16 route: groups 2c and 2c+1
    float fA_lo = 0.0f, fA_hi = 0.0f, fB_lo = 0.0f, fB_hi = 0.0f;
    if (F16) {
        const uint32_t pa = e4m3x2_to_f16x2(sa & 0xFFFFu);
        const uint32_t pb = e4m3x2_to_f16x2(sb & 0xFFFFu);
        const __half2 ha = *reinterpret_cast<const __half2 *>(&pa);
        const __half2 hb = *reinterpret_cast<const __half2 *>(&pb);
        scA_lo = __low2half2(ha);
        scA_hi = __high2half2(ha);
        scB_lo = __low2half2(hb);
        scB_hi = __high2half2(hb);
    } else if (GS == 16) {
        fA_lo = e4m3_to_f32(sa & 0xFFu);
        fA_hi = e4m3_to_f32((sa >> 8) & 0xFFu);
        fB_lo = e4m3_to_f32(sb & 0xFFu);
        fB_hi = e4m3_to_f32((sb >> 8) & 0xFFu);
    } else {
        fA_lo = fA_hi = e8m0_to_f32(sa & 0xFFu);
        fB_lo = fB_hi = e8m0_to_f32(sb & 0xFFu);
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
    const uint16_t *const bro_t[2] = {bro + 4 * swz, bro + 4 * (swz ^ 1)};
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
            const int sh = GS == 16 ? 16 * h : 8 * h;
            mma_block<GS, F16>(d, wa[h], wb[h], sa >> sh, sb >> sh, bro_t, 2 * b + h);
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
        decode_prologue<kDecThreads>(p, c0, rows, act, ascale, rowscale, rowok, route_f16,
                                     write_codes);
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

// ---------------------------------------------------------------- TMA-fed decode kernel
//
// The same MMA work as decode_mma_kernel, with the weights brought in by TMA instead of
// per-lane loads, so that the bytes in flight per SM are set by a shared-memory ring and
// not by registers. Persistent: one CTA per SM takes a contiguous run of the call's items
// (expert, pass of up to PR routed rows, 128-row weight block), in expert order, so a CTA
// quantises a pass's activation rows once for all its consecutive items of that pass.
//   warps 0 .. CW-1  consumers: act_quant prologue at each new (expert, pass), then per
//                    ring stage the MMAs of their 16 weight rows (mma_block), outputs per
//                    item. With CW = 16, warps w and w + 8 share rows and split each
//                    stage's four 128-k blocks (w takes blocks 0 and 2, w + 8 blocks 1 and
//                    3); w + 8 hands its partial sums to w through shared memory.
//   warp CW          producer: per stage, two 128-row x 128-byte nibble boxes (512 k,
//                    128-byte swizzle) and the stage's scale box, into an S-slot ring
// Each warp keeps CH accumulators and sends its successive blocks to them in turn (CH
// independent MMA chains), adding them in order at the end of the item.
// The fragment rows of a warp are permuted (fragment row g reads weight row
// (g >> 1) + 4 (g & 1) of its eight) so that the eight lanes of a shared-memory phase read
// rows r and r + 4, whose 16-byte chunks the swizzle puts in opposite halves of the
// 128-byte line: every 16-byte read of a warp is conflict-free.
namespace dtma {
constexpr int BM = kDecCols;                          // weight rows per item
constexpr int KS = 512;                               // k per ring stage
constexpr int NIB_BOX = BM * 128;                     // 128 rows x 128 bytes (256 k)
constexpr int SC_ROW_MAX = KS / 16;                   // scale bytes per row and stage (NVFP4)
constexpr int STAGE_BYTES = 2 * NIB_BOX + BM * SC_ROW_MAX;
constexpr int kMaxStages = 6;
constexpr int kMinStages = 3;
constexpr int kMaxExperts = 1024;
constexpr int kPairBarrier = 2;                       // named barriers 2 .. 9: warp pairs
constexpr int kPassCache = 8;                         // passes whose token ids are cached
// Stages a producer keeps in flight (issued, not landed). On GB300 a read stream through
// TMA reaches its peak with about 64 KB in flight per SM; more only lengthens the memory
// queue, and with it the wait of every other read (the activation rows of a prologue).
constexpr int kInFlight = 2;
// the configuration the library launches: consumer warps and accumulator chains per warp
constexpr int kWarps = 16;
constexpr int kChains = 2;
static_assert(STAGE_BYTES % 1024 == 0 && NIB_BOX % 1024 == 0, "swizzled boxes need 1024-byte alignment");
} // namespace dtma

struct DtmaLayout {
    int stages;
    size_t act, ascale, rowscale, rowok, route, xbuf, bars, prefix, offs, sc2, ptok, npc, flag,
        total;
};

// Bounded wait taken by lane 0 for the whole warp, so that the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned *err)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0)
        ok = mbar_wait(bar, parity, abort_flag, err);
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

// Multiprocessor count of the current device, looked up once per device.
static int decode_sms()
{
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 152;
    if (cached[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            sms = 152;
        cached[dev] = sms;
    }
    return cached[dev];
}

// Shared memory of decode_tma_kernel for PR rows per pass, or stages = 0 if fewer than
// kMinStages ring slots fit.
static DtmaLayout dtma_layout(int pr, int64_t k, int E)
{
    using namespace dtma;
    DtmaLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) {
        off = (off + align - 1) / align * align;
        const size_t at = off;
        off += bytes;
        return at;
    };
    L.act = take((size_t)pr * (k + kDecRowPad) * 2, 16);
    L.ascale = take((size_t)pr * (k / 128) * 4, 16);
    L.rowscale = take((size_t)pr * 4, 4);
    L.rowok = take((size_t)pr * 4, 4);
    L.route = take(4, 4);
    L.xbuf = take(2 * 8 * 32 * 4 * 4, 16);  // [item parity][warp pair][lane][4] partial sums
    L.bars = take(2 * kMaxStages * 8, 8);
    L.prefix = take(((size_t)E + 1) * 4, 4);
    L.offs = take(((size_t)E + 1) * 4, 4);
    L.sc2 = take((size_t)E * 4, 4);
    L.ptok = take((size_t)kPassCache * pr * 4, 4);
    L.npc = take(4, 4);
    L.flag = take(4, 4);
    const size_t fixed = (off + 1023) / 1024 * 1024;
    // 1024: alignment slack of the dynamic shared-memory base
    const size_t room = fixed + 1024 < kDecSmemLimit ? kDecSmemLimit - 1024 - fixed : 0;
    L.stages = (int)std::min<size_t>(kMaxStages, room / STAGE_BYTES);
    if (L.stages < kMinStages)
        L.stages = 0;
    L.total = 1024 + (size_t)L.stages * STAGE_BYTES + fixed;
    return L;
}


struct DtmaParams {
    GroupedProblem p;
    DtmaLayout L;
    int mt;  // 128-row weight blocks per expert
};

template <int GS, int PR, int CW, int CH>
__global__ void __launch_bounds__((CW + 1) * 32, 1)
    decode_tma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                      const DtmaParams dp)
{
    using namespace dtma;
    static_assert(CW == 8 || CW == 16, "consumer warps");
    static_assert(CH == 1 || CH == 2, "accumulator chains");
    constexpr int NT = CW * 32;       // consumer threads
    constexpr int NG = CW / 8;        // warp groups splitting a stage's blocks
    constexpr int kThreads = NT + 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const GroupedProblem &p = dp.p;
    const DtmaLayout &L = dp.L;
    const int S = L.stages;
    uint8_t *ring = base;
    uint8_t *fixed = base + (size_t)S * STAGE_BYTES;
    uint16_t *act = reinterpret_cast<uint16_t *>(fixed + L.act);
    float *ascale = reinterpret_cast<float *>(fixed + L.ascale);
    float *rowscale = reinterpret_cast<float *>(fixed + L.rowscale);
    int *rowok = reinterpret_cast<int *>(fixed + L.rowok);
    int *route_f16 = reinterpret_cast<int *>(fixed + L.route);
    float4 *xbuf = reinterpret_cast<float4 *>(fixed + L.xbuf);
    uint64_t *bars = reinterpret_cast<uint64_t *>(fixed + L.bars);
    int *prefix = reinterpret_cast<int *>(fixed + L.prefix);
    int32_t *offs = reinterpret_cast<int32_t *>(fixed + L.offs);
    float *sc2 = reinterpret_cast<float *>(fixed + L.sc2);
    int32_t *ptok = reinterpret_cast<int32_t *>(fixed + L.ptok);
    int *npc = reinterpret_cast<int *>(fixed + L.npc);  // passes whose token ids are cached
    volatile int *abort_flag = reinterpret_cast<volatile int *>(fixed + L.flag);
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };

    const int k = p.k, n = p.n, E = p.E, mt = dp.mt;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Launched with programmatic stream serialization: a kernel queued behind this one may
    // be scheduled as this one's CTAs exit, and this one may start while the kernel before
    // it drains. Nothing of global memory is read before that kernel has completed and its
    // writes are visible (griddepcontrol.wait), so any input may come from it.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // items per expert: passes of up to PR rows x weight blocks (bad offsets: none); the
    // offsets stay in shared memory (reads of global memory behind the weight stream wait
    // for the whole memory queue)
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int64_t r0 = 0, r1 = p.P;
        if (p.offsets) {
            r0 = p.offsets[e];
            r1 = p.offsets[e + 1];
        }
        offs[e] = (int32_t)r0;
        if (e == E - 1)
            offs[E] = (int32_t)r1;
        sc2[e] = (GS == 16) ? (p.scale2 ? p.scale2[e] : p.scale2_host) : 1.0f;
        const bool bad = r0 < 0 || r1 < r0 || r1 > p.P || (e == 0 && r0 != 0) ||
                         (e == E - 1 && r1 != p.P);
        int cnt = 0;
        if (bad) {
            if (blockIdx.x == 0)
                raise_device_error(p.err, FP4_DEVERR_OFFSETS);
        } else {
            cnt = (int)((r1 - r0 + PR - 1) / PR) * mt;
        }
        prefix[e + 1] = cnt;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), CW);
        }
        prefix[0] = 0;
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0) {  // prefix scan: each lane sums a contiguous chunk, then a warp scan
        const int per = (E + 31) / 32;
        const int lo = 1 + lane * per, hi = min(E + 1, lo + per);
        int run = 0;
        for (int i = lo; i < hi; ++i)
            run += prefix[i];
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += v;
        }
        int acc = incl - run;
        for (int i = lo; i < hi; ++i) {
            acc += prefix[i];
            prefix[i] = acc;
        }
    }
    __syncthreads();
    const int total = prefix[E];
    const int t0 = (int)(((int64_t)total * blockIdx.x) / gridDim.x);
    const int t1 = (int)(((int64_t)total * (blockIdx.x + 1)) / gridDim.x);
    const int nst = k / KS;
    // item t -> expert, pass, weight block
    auto item = [&](int t, int &e, int &pass, int &m) {
        int lo = 0, hi = E;  // prefix[lo] <= t < prefix[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= t)
                lo = mid;
            else
                hi = mid;
        }
        e = lo;
        const int local = t - prefix[lo];
        pass = local / mt;
        m = local - pass * mt;
    };
    // Steps through this CTA's items in order from t0, reading the prefix only where the
    // expert changes (a shared-memory read behind the consumers' operand traffic costs a
    // few hundred cycles, and the item boundary holds up every consumer warp).
    struct Walk {
        int e, pass, m, end;  // end: the first item past expert e
    };
    auto walk_start = [&](Walk &w) {
        item(t0, w.e, w.pass, w.m);
        w.end = prefix[w.e + 1];
    };
    auto walk_next = [&](Walk &w, int t) {
        if (++w.m == mt) {
            w.m = 0;
            ++w.pass;
        }
        if (t >= w.end) {
            do {
                ++w.e;
                w.end = prefix[w.e + 1];
            } while (t >= w.end);
            w.pass = 0;
            w.m = 0;
        }
    };

    if (warp == CW) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            constexpr uint32_t tx = 2 * NIB_BOX + BM * (KS / GS);
            // weights are read once: evict them from L2 first (measured on GB300: a read
            // stream through TMA reaches about 0.92 of the copy bandwidth with this hint,
            // 0.82 without)
            const uint64_t policy = l2_evict_first_policy();
            int slot = 0, oslot = 0, inflight = 0;  // oslot: the oldest stage still in flight
            uint32_t phase = 0, ophase = 0, issued = 0, parity = 0;
            bool ok = true;
            Walk wk;
            if (t0 < t1)
                walk_start(wk);
            for (int t = t0; t < t1 && ok; ++t) {
                if (t > t0)
                    walk_next(wk, t);
                const int y = wk.e * n + wk.m * BM;
                for (int j = 0; j < nst; ++j) {
                    if (inflight == kInFlight) {
                        if (!mbar_wait(full(oslot), ophase, abort_flag, p.err)) {
                            ok = false;
                            break;
                        }
                        --inflight;
                        if (++oslot == S) {
                            oslot = 0;
                            ophase ^= 1u;
                        }
                    }
                    if (!mbar_wait(empty(slot), phase ^ 1u, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dst = ring + (size_t)slot * STAGE_BYTES;
                    const uint32_t fb = full(slot);
                    mbar_arrive_expect_tx(fb, tx);
                    const uint32_t d0 = (uint32_t)__cvta_generic_to_shared(dst);
                    tma_load_2d_evict_first(d0, &tmW, j * (KS / 2), y, fb, policy);
                    tma_load_2d_evict_first(d0 + NIB_BOX, &tmW, j * (KS / 2) + 128, y, fb, policy);
                    tma_load_2d_evict_first(d0 + 2 * NIB_BOX, &tmS, j * (KS / GS), y, fb, policy);
                    issued |= 1u << slot;
                    parity = (parity & ~(1u << slot)) | (phase << slot);
                    ++inflight;
                    if (++slot == S) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {  // let this CTA's own copies land before it exits
                for (int s = 0; s < S; ++s)
                    if (issued & (1u << s))
                        mbar_drain(full(s), (parity >> s) & 1u);
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    if (warp == 0) {
        // the token ids of this CTA's first kPassCache passes into shared memory, and their
        // activation rows into L2, before the weight stream fills the memory queue. Lane l
        // looks at item t0 + l; a pass starts where (expert, pass) changes.
        const int t = t0 + lane;
        int e = -1, pass = -1, m = 0;
        if (t < t1)
            item(t, e, pass, m);
        const int pe = __shfl_up_sync(0xFFFFFFFFu, e, 1), pp = __shfl_up_sync(0xFFFFFFFFu, pass, 1);
        const bool start = t < t1 && (lane == 0 || e != pe || pass != pp);
        const unsigned starts = __ballot_sync(0xFFFFFFFFu, start);
        const int pi = __popc(starts & ((2u << lane) - 1u)) - 1;  // this lane's pass index
        if (lane == 0)
            *npc = min(__popc(starts), kPassCache);
        if (start && pi < kPassCache) {
            const int64_t c0 = (int64_t)offs[e] + (int64_t)pass * PR;
            const int rows = (int)min((int64_t)PR, (int64_t)offs[e + 1] - c0);
            for (int r = 0; r < PR; ++r) {
                int32_t tok = -1;
                if (r < rows) {
                    tok = p.row_ids ? p.row_ids[c0 + r] : (int32_t)(c0 + r);
                    if (tok >= 0 && tok < p.T)
                        prefetch_l2(p.x + (int64_t)tok * k, (uint32_t)k * 4u);
                }
                ptok[pi * PR + r] = tok;
            }
        }
    }
    const int rw = warp & 7, grp = warp >> 3;  // row block of 16, block group
    const int g = lane >> 2, c = lane & 3, swz = c >> 1;
    const int rA = rw * kDecRowsPerWarp + (g >> 1) + 4 * (g & 1), rB = rA + 8;
    const int ld = k + kDecRowPad;
    const uint16_t *bro = act + (size_t)min(g, PR - 1) * ld + 32 * c;
    const uint16_t *const bro_t[2] = {bro + 4 * swz, bro + 4 * (swz ^ 1)};
    // this lane's 16-byte chunk of block h (0..3) of a stage, rows rA and rB: box h / 2,
    // logical chunk 4 (h & 1) + c at physical chunk (logical ^ (row & 7)); rA & 7 == rB & 7
    auto choff = [&](int h) { return (h >> 1) * NIB_BOX + ((((h & 1) << 2 | c) ^ (rA & 7)) << 4); };
    constexpr int SCR = KS / GS;  // scale bytes per row and stage
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    int prev_e = -1, prev_pass = -1, npass = 0;
    int64_t c0 = 0;
    int rows = 0;
    float s2 = 1.0f;
    bool f16 = false;
    // the pass's values this lane's output columns 2c, 2c + 1 need, kept in registers
    bool col_ok[2] = {false, false};
    float col_rs[2] = {1.0f, 1.0f};
    Walk wk;
    if (t0 < t1)
        walk_start(wk);
    for (int t = t0; t < t1; ++t) {
        if (t > t0)
            walk_next(wk, t);
        const int e = wk.e, pass = wk.pass, m = wk.m;
        if (e != prev_e || pass != prev_pass) {
            consumer_sync<NT>();  // every consumer is done with the previous pass's rows
            const int64_t r0 = offs[e], r1 = offs[e + 1];
            c0 = r0 + (int64_t)pass * PR;
            rows = (int)((r1 - c0) < PR ? (r1 - c0) : PR);
            s2 = sc2[e];
            decode_prologue<NT>(p, c0, rows, act, ascale, rowscale, rowok, route_f16,
                                p.codes_out != nullptr && m == 0,
                                npass < *npc ? ptok + npass * PR : nullptr);
            prev_e = e;
            prev_pass = pass;
            ++npass;
            f16 = GS == 16 && *route_f16 != 0;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int nn = 2 * c + q;
                col_ok[q] = nn < rows && rowok[nn] != 0;
                col_rs[q] = col_ok[q] && f16 ? rowscale[nn] : 1.0f;
            }
        }
        float d[CH][4];
#pragma unroll
        for (int ch = 0; ch < CH; ++ch)
            d[ch][0] = d[ch][1] = d[ch][2] = d[ch][3] = 0.0f;
        for (int j = 0; j < nst; ++j) {
            if (ok)
                ok = warp_wait(full(slot), phase, abort_flag, p.err);
            if (ok) {
                const uint8_t *st = ring + (size_t)slot * STAGE_BYTES;
                const uint8_t *scA = st + 2 * NIB_BOX + rA * SCR;
                const uint8_t *scB = st + 2 * NIB_BOX + rB * SCR;
#pragma unroll
                for (int i = 0; i < 4 / NG; ++i) {
                    const int h = grp + NG * i;
                    const uint4 wa = *reinterpret_cast<const uint4 *>(st + rA * 128 + choff(h));
                    const uint4 wb = *reinterpret_cast<const uint4 *>(st + rB * 128 + choff(h));
                    uint32_t sa, sb;
                    if (GS == 16) {  // groups 8h + 2c, 8h + 2c + 1
                        sa = *reinterpret_cast<const uint16_t *>(scA + 8 * h + 2 * c);
                        sb = *reinterpret_cast<const uint16_t *>(scB + 8 * h + 2 * c);
                    } else {  // group 4h + c
                        sa = scA[4 * h + c];
                        sb = scB[4 * h + c];
                    }
                    float(&dc)[4] = d[i % CH];
                    if (f16)
                        mma_block<GS, true>(dc, wa, wb, sa, sb, bro_t, 4 * j + h);
                    else
                        mma_block<GS, false>(dc, wa, wb, sa, sb, bro_t, 4 * j + h);
                }
                // the stage's values are consumed (the MMAs used them): release the slot,
                // behind an async-proxy fence that orders these reads before the refill
                fence_proxy_async();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty(slot));
            }
            if (++slot == S) {
                slot = 0;
                phase ^= 1u;
            }
        }
        // the warp's sum: its chains in order
        float r[4] = {d[0][0], d[0][1], d[0][2], d[0][3]};
        if (CH == 2) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                r[q] += d[CH - 1][q];
        }
        if (NG == 2) {
            // warp rw + 8 hands its sums to warp rw (double-buffered by item parity; the
            // pair barrier of item i + 1 orders the read of item i before the next write)
            float4 *xb = xbuf + ((size_t)(t & 1) * 8 + rw) * 32 + lane;
            if (grp == 1)
                *xb = make_float4(r[0], r[1], r[2], r[3]);
            named_sync(kPairBarrier + rw, 64);
            if (grp == 1)
                continue;
            const float4 o = *xb;
            r[0] += o.x;
            r[1] += o.y;
            r[2] += o.z;
            r[3] += o.w;
        }
        if (!ok)
            continue;  // aborting: the barrier sequence above is kept, nothing is stored
        // D: (fragment row g, n = 2c, 2c+1) in r0, r1; (fragment row g + 8) in r2, r3
        const int colA = m * BM + rA, colB = m * BM + rB;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int q = jj & 1;
            const int col = (jj < 2) ? colA : colB;
            if (col_ok[q] && col < n)
                p.out[(c0 + 2 * c + q) * (int64_t)n + col] = (r[jj] * col_rs[q]) * s2;
        }
    }
}

// Whether decode_tma_kernel takes this call: k a whole number of 512-k stages, at most
// kMaxExperts experts, the ring fits next to PR activation rows, TMA-aligned weights.
static bool dtma_ok(const GroupedProblem &p, int pr)
{
    using namespace dtma;
    if (p.k % KS != 0 || p.E > kMaxExperts || (int64_t)p.E * p.n >= ((int64_t)1 << 31))
        return false;
    if ((reinterpret_cast<uintptr_t>(p.w) & 15) || (reinterpret_cast<uintptr_t>(p.sc) & 15))
        return false;
    return dtma_layout(pr, p.k, p.E).stages > 0;
}

template <int GS, int PR>
static cudaError_t launch_dtma(const GroupedProblem &p, cudaStream_t s)
{
    using namespace dtma;
    DtmaParams dp;
    dp.p = p;
    dp.L = dtma_layout(PR, p.k, p.E);
    dp.mt = (p.n + BM - 1) / BM;
    alignas(64) CUtensorMap tmW, tmS;
    if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w, (uint64_t)p.k / 2,
                  (uint64_t)p.E * p.n, 128, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.sc, (uint64_t)p.k / GS,
                  (uint64_t)p.E * p.n, KS / GS, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    auto kern = decode_tma_kernel<GS, PR, kWarps, kChains>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kDecSmemLimit);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            attr_set[dev] = true;
    }
    // an upper bound of the items (every expert's rows in whole passes); the kernel splits
    // the exact count evenly over the CTAs it gets
    const int64_t max_items = ((p.P + PR - 1) / PR + p.E) * (int64_t)dp.mt;
    const int grid = (int)std::min<int64_t>(max_items, decode_sms());
    // programmatic stream serialization: the launch latency and CTA start-up of this kernel
    // overlap the tail of the previous one on the stream (measured on GB300: 3 us per
    // gate/up + down decode step); the kernel waits for that one's completion before it
    // reads global memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((kWarps + 1) * 32);
    cfg.dynamicSmemBytes = dp.L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmW, tmS, dp);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

static size_t decode_smem_bytes(int pr, int64_t k)
{
    return (size_t)pr * (k + kDecRowPad) * 2 + (size_t)pr * (k / 128) * 4 + (size_t)pr * 8 + 16;
}

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
    const int pr = rows_per_pass <= 4 || !dtma_ok(p, 8) ? 4 : 8;
    if (dtma_ok(p, pr)) {
        if (pr == 4)
            return nv ? launch_dtma<16, 4>(p, s) : launch_dtma<32, 4>(p, s);
        return nv ? launch_dtma<16, 8>(p, s) : launch_dtma<32, 8>(p, s);
    }
    if (rows_per_pass <= 4 || decode_smem_bytes(8, p.k) > kDecSmemLimit)
        return nv ? launch_pr<16, 4>(p, s) : launch_pr<32, 4>(p, s);
    return nv ? launch_pr<16, 8>(p, s) : launch_pr<32, 8>(p, s);
}

// One f32 accumulation per k16 MMA step, the row-scale multiply (exact) and the scale2
// multiply; NVFP4 adds the f32 rounding of ws = e4m3 * scale2 that the f64 reference takes
// where this path multiplies by scale2 last, and that of the final product. (The TMA-fed
// kernel splits the k16 steps over four chains, k/64 each, and adds the chains in two
// levels: k/64 + 2 roundings on any term's path, within the k/16 counted here.)
double decode_error_ops(int recipe, int64_t k)
{
    return (double)(k / 16) + (recipe == FP4_NVFP4 ? 2.0 : 0.0) + 1.0;
}

} // namespace fp4moe
