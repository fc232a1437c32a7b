// gemm_stream.cu -- weight-streaming grouped expert GEMM on CUDA cores, act_quant fused.
//
// The no-workspace path for k too long for the warp-MMA decode kernel's shared memory
// (four activation rows of k > 28544). Like that kernel it is bound by HBM reads of the
// nibble weights (0.5 B per weight plus 1/16 or 1/32 B of scale). It streams every
// touched expert's weights once with 128-bit loads and keeps the arithmetic on CUDA
// cores in the order the pages define (fn mirror_gemm / fn f64_ref of memra-engine
// 0.98.0, src/bin/dsv4_native_gemm_gate.rs):
//   sub  = sum over the gs weights of a group of e4m3(a) * E2M1(w)   (exact products,
//          f32 adds; f16 operands through fma.rn.f32.f16)
//   ws   = f32(e4m3(scale) * scale2)  (NVFP4)   or  2^(e-127)  (MXFP4)
//   acc  = fma(sub, ws * s_act, acc)
// then a warp-shuffle sum over the 32 lanes that split k.
//
// Layout: CTA (256 threads) = one expert x 64 output columns (weight rows); warp w owns
// 8 weight rows; lane l reads k in chunks [32 l + 1024 i, +32): 16 B of nibbles per
// weight row per chunk, so a warp reads 512 contiguous bytes of each row per step.
// Activation rows of the expert are quantised by the CTA in a prologue (fused
// act_quant), up to 2 rows a pass (what shared memory holds at these k), into shared
// memory as exact f16 code values plus the per-128 f32 scales; the weights of the CTA are
// re-read (from L2) once per pass. Each pass runs code specialised for its row count, so
// an expert with one routed row does one row's arithmetic.
#include "common.cuh"

#include <algorithm>

namespace fp4moe {

constexpr int kStreamThreads = 256;
constexpr int kRowsPerWarp = 8;
constexpr int kColsPerCta = (kStreamThreads / 32) * kRowsPerWarp;

template <int RB>
__device__ __forceinline__ void quantize_chunk(const GroupedProblem &p, int64_t c0, int rows,
                                               __half *act, float *ascale, int *rowok,
                                               bool write_codes)
{
    const int k = p.k, kq = k >> 7;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int gi = warp; gi < RB * kq; gi += kStreamThreads / 32) {
        const int r = gi / kq, g = gi - r * kq;
        uint2 h = make_uint2(0u, 0u);
        float s = 0.0f;
        int ok = 0;
        if (r < rows) {
            const int64_t pr = c0 + r;
            const int64_t t = p.row_ids ? (int64_t)p.row_ids[pr] : pr;
            if (t >= 0 && t < p.T) {
                ok = 1;
                const float4 v =
                    *reinterpret_cast<const float4 *>(p.x + t * (int64_t)k + g * 128 + lane * 4);
                float amax =
                    fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
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
        }
        *reinterpret_cast<uint2 *>(act + (size_t)r * k + g * 128 + lane * 4) = h;
        if (lane == 0) {
            ascale[r * kq + g] = s;
            if (g == 0)
                rowok[r] = ok;
        }
    }
}

// Weights and scales of one 32-wide k chunk for the warp's 8 weight rows.
template <int GS>
__device__ __forceinline__ void load_chunk(const uint8_t *wexp, const uint8_t *sexp, size_t wrow,
                                           size_t srow, int col_base, int n, int kb,
                                           uint4 (&wv)[kRowsPerWarp],
                                           uint32_t (&sb)[kRowsPerWarp])
{
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int col = col_base + i;
        if (col < n) {
            wv[i] = ld_stream_v4(wexp + (size_t)col * wrow + (kb >> 1));
            if (GS == 16)
                sb[i] = *reinterpret_cast<const uint16_t *>(sexp + (size_t)col * srow + (kb >> 4));
            else
                sb[i] = sexp[(size_t)col * srow + (kb >> 5)];
        } else {
            wv[i] = make_uint4(0u, 0u, 0u, 0u);
            sb[i] = 0u;
        }
    }
}

// One pass over the CTA's weight rows for RB quantised activation rows in shared memory.
template <int RB, int GS>
__device__ __forceinline__ void stream_pass(const GroupedProblem &p, const __half *act,
                                            const float *ascale, const int *rowok, int64_t c0,
                                            int rows, const uint8_t *wexp, const uint8_t *sexp,
                                            int col_base, float s2)
{
    const int k = p.k, n = p.n, kq = k >> 7;
    const int lane = threadIdx.x & 31;
    const size_t wrow = (size_t)k / 2, srow = (size_t)k / GS;

    float acc[kRowsPerWarp][RB];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
        for (int r = 0; r < RB; ++r)
            acc[i][r] = 0.0f;

    for (int kb = lane * 32; kb < k; kb += 1024) {
        uint4 wv[kRowsPerWarp];
        uint32_t sb[kRowsPerWarp];
        load_chunk<GS>(wexp, sexp, wrow, srow, col_base, n, kb, wv, sb);
        float asv[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r)
            asv[r] = ascale[r * kq + (kb >> 7)];

        float subm[kRowsPerWarp][RB];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t a[RB][8];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const uint4 *ap = reinterpret_cast<const uint4 *>(act + (size_t)r * k + kb + 16 * h);
                const uint4 a0 = ap[0], a1 = ap[1];
                a[r][0] = a0.x; a[r][1] = a0.y; a[r][2] = a0.z; a[r][3] = a0.w;
                a[r][4] = a1.x; a[r][5] = a1.y; a[r][6] = a1.z; a[r][7] = a1.w;
            }
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                uint32_t wh[8];
                uint32_t lo[4], hi[4];
                e2m1x8_to_f16x8(h ? wv[i].z : wv[i].x, lo);
                e2m1x8_to_f16x8(h ? wv[i].w : wv[i].y, hi);
                wh[0] = lo[0]; wh[1] = lo[1]; wh[2] = lo[2]; wh[3] = lo[3];
                wh[4] = hi[0]; wh[5] = hi[1]; wh[6] = hi[2]; wh[7] = hi[3];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    float sub = (GS == 32 && h == 1) ? subm[i][r] : 0.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        sub = fma2_f16_f32(wh[j], a[r][j], sub);
                    if (GS == 16) {
                        const float ws = e4m3_to_f32((sb[i] >> (8 * h)) & 0xFFu) * s2;
                        acc[i][r] = fmaf(sub, ws * asv[r], acc[i][r]);
                    } else if (h == 1) {
                        const float ws = e8m0_to_f32(sb[i]);
                        acc[i][r] = fmaf(sub, ws * asv[r], acc[i][r]);
                    } else {
                        subm[i][r] = sub;
                    }
                }
            }
        }
    }

    // Reduce over the 32 lanes; lane i ends up writing column col_base + i.
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        float mine = 0.0f;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const float v = warp_sum(acc[i][r]);
            if (lane == i)
                mine = v;
        }
        if (r < rows && lane < kRowsPerWarp && col_base + lane < n && rowok[r])
            p.out[(c0 + r) * (int64_t)n + col_base + lane] = mine;
    }
}

// Quantise the next `rows` (= RB) activation rows into shared memory, then stream.
template <int RB, int GS>
__device__ __forceinline__ void stream_rows(const GroupedProblem &p, __half *act, float *ascale,
                                            int *rowok, int64_t c0, const uint8_t *wexp,
                                            const uint8_t *sexp, int col_base, float s2,
                                            bool write_codes)
{
    __syncthreads();
    quantize_chunk<RB>(p, c0, RB, act, ascale, rowok, write_codes);
    __syncthreads();
    stream_pass<RB, GS>(p, act, ascale, rowok, c0, RB, wexp, sexp, col_base, s2);
}

// RBMAX: most activation rows the shared-memory buffer holds (by k). Each pass takes
// min(rows left, RBMAX) rows with code specialised for that count, so an expert with one
// routed row does one row's arithmetic, and an expert with up to RBMAX rows reads its
// weights once.
template <int RBMAX, int GS>
__global__ void __launch_bounds__(kStreamThreads, 2) stream_gemm_kernel(const GroupedProblem p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int k = p.k, n = p.n, kq = k >> 7;
    __half *act = reinterpret_cast<__half *>(smem);
    float *ascale = reinterpret_cast<float *>(smem + (size_t)RBMAX * k * 2);
    int *rowok = reinterpret_cast<int *>(ascale + RBMAX * kq);

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

    const int warp = threadIdx.x >> 5;
    const int col_base = blockIdx.x * kColsPerCta + warp * kRowsPerWarp;
    const float s2 = (GS == 16) ? (p.scale2 ? p.scale2[e] : p.scale2_host) : 1.0f;
    const uint8_t *wexp = p.w + (size_t)e * n * ((size_t)k / 2);
    const uint8_t *sexp = p.sc + (size_t)e * n * ((size_t)k / GS);
    const bool write_codes = p.codes_out != nullptr && blockIdx.x == 0;

    for (int64_t c0 = r0; c0 < r1;) {
        const int left = (int)((r1 - c0) < RBMAX ? (r1 - c0) : RBMAX);
        if (RBMAX >= 2 && left == 2) {
            stream_rows<(RBMAX >= 2 ? 2 : 1), GS>(p, act, ascale, rowok, c0, wexp, sexp, col_base,
                                                   s2, write_codes);
            c0 += 2;
        } else {
            stream_rows<1, GS>(p, act, ascale, rowok, c0, wexp, sexp, col_base, s2, write_codes);
            c0 += 1;
        }
    }
}

static size_t stream_smem_bytes(int rb, int k)
{
    return (size_t)rb * k * 2 + (size_t)rb * (k / 128) * 4 + (size_t)rb * 4;
}

template <int RBMAX, int GS>
static cudaError_t launch_rb(const GroupedProblem &p, cudaStream_t s)
{
    const size_t smem = stream_smem_bytes(RBMAX, p.k);
    auto kern = stream_gemm_kernel<RBMAX, GS>;
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    dim3 grid((unsigned)((p.n + kColsPerCta - 1) / kColsPerCta), (unsigned)p.E);
    kern<<<grid, kStreamThreads, smem, s>>>(p);
    return cudaGetLastError();
}

int stream_max_rows_per_pass(int k)
{
    const size_t limit = 227 * 1024;
    for (int rb : {2, 1})
        if (stream_smem_bytes(rb, k) <= limit)
            return rb;
    return 0;
}

cudaError_t launch_stream_gemm(const GroupedProblem &p, int rows_per_pass, cudaStream_t s)
{
    const int rb = std::min(rows_per_pass, stream_max_rows_per_pass(p.k));
    const bool nv = p.recipe == FP4_NVFP4;
    switch (rb) {
    case 2: return nv ? launch_rb<2, 16>(p, s) : launch_rb<2, 32>(p, s);
    case 1: return nv ? launch_rb<1, 16>(p, s) : launch_rb<1, 32>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

// Summation depth of one output: (gs - 1) rounded adds inside a group, one fused
// multiply-add per group a lane visits (2 groups per 32-wide chunk for NVFP4, 1 for
// MXFP4, ceil(k/1024) chunks), then 5 shuffle-tree levels. The NVFP4 ws = e4m3*scale2
// rounding is the one the f64 reference also takes, so it adds nothing.
double stream_error_ops(int recipe, int64_t k)
{
    const int gs = recipe == FP4_NVFP4 ? 16 : 32;
    const int64_t chunks = (k + 1023) / 1024;
    const int64_t groups_per_lane = (recipe == FP4_NVFP4 ? 2 : 1) * chunks;
    return (double)(gs - 1) + (double)groups_per_lane + 5.0;
}

} // namespace fp4moe
