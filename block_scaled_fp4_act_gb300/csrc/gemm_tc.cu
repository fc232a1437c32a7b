// gemm_tc.cu -- NVFP4 tensor-core grouped expert GEMM for prefill-sized row counts
// (sm_103a: TMA, mbarrier pipeline, tcgen05.mma with the accumulator in tensor memory),
// its quantise pass, and the allocation-free entry point.
//
// Arithmetic (memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs, fn f64_ref): every
// product e4m3(a) * s_a * E2M1(w) * ws is formed exactly and summed in f32. The MMA
// kind that accepts FP8 operands has only ue8m0 scales per 32, and the kind with e4m3
// scales per 16 wants FP4 on both sides, so the exact route for NVFP4 on this hardware is
// the 16-bit MMA (kind::f16): both operands carry their scales and stay exact.
//   A (M side) = weights:     f16(E2M1 * e4m3 scale) on the f16 route, bf16 otherwise
//                             (<= 6 significant bits either way)
//   B (N side) = activations: f16(code * 2^(m - M)) or bf16(code * 2^m), written by the
//                             quantise pass (M: the routed row's largest block exponent)
//   D (TMEM)   = f32 [128 weight rows x N routed rows]; the epilogue multiplies by the
//                row scale 2^M (f16 route) and scale2.
// (MXFP4 runs on the block-scaled 8-bit MMA instead: gemm_mx.cu.)
//
// Kernel structure: persistent, one CTA (24 warps) per SM, static round-robin over
// tiles (expert, 192-row block of its routed rows, 128-row block of its weights),
// weight-row block fastest so consecutive tiles share the activation block in L2.
// Rings decouple the streams: a 4-slot shared-memory weight ring (each slot 256 k of the
// tile's 128 weight rows: 128-byte nibble lines in the 128-byte swizzle + 16 scale bytes
// per row; the weights stream from HBM once per tile), a 6-slot activation ring in shared
// memory and a 4-stage ring of converted 64-k weight stages in tensor memory, from which
// the MMA reads its A operand.
//   warp 0      TMA producer of activation slots (16-bit, 128B swizzle, k-block-major)
//   warp 1      TMEM owner and MMA issuer (whole warp, one elected lane issues), 4 MMAs
//               of K=16 per stage
//   warp 2      TMA producer of the weight slots (nibble box + scale box)
//   warp 3      relay: does the MMA side's mbarrier waits and releases each A stage to
//               warp 1 through a hardware named barrier
//   warps 4-7   epilogue: tcgen05.ld of the accumulator, x row scale x scale2; whole
//               32-row chunks staged in shared memory and written by one bulk tensor
//               store each, the rest (and SwiGLU's h) by coalesced f32 stores
//   warps 8-23  converters, four per TMEM lane quarter taking turns over the k-stages:
//               nibbles x scales -> 16-bit A operand, tcgen05.st into TMEM
// Two accumulators (2 x 192 TMEM columns) let the epilogue of one tile overlap the
// main loop of the next. The MMA N of a tile is its routed-row count rounded up to 16,
// so an expert's ragged last block costs at most 15 padded rows.
//
// The MMA warp touches no mbarrier and no shared memory inside a tile. A wait or load
// issued behind queued MMAs completes only once those MMAs have been handed to the tensor
// core, so a per-stage mbarrier wait in the issuing warp idles the tensor pipe for about
// 130 cycles a stage (measured on GB300: 340 cycles per 4-MMA stage at N <= 128 against
// 256 without it). The relay warp takes those waits and passes readiness on with
// bar.arrive / bar.sync, which do not go through that queue.
//
// Every mbarrier wait is bounded (about a second of clock64 cycles, or the shorter limit
// of a test launch); on expiry the CTA sets the TIMEOUT bit of the device error word,
// stops all roles, waits (bounded) for its own copies and MMAs in flight, frees its
// tensor memory and returns. The MMA warp's named-barrier waits cannot time out, so on
// abort the relay keeps releasing stages to the end of the current tile, each only after
// the MMA warp has consumed the slot's previous use (a bounded wait on the slot's empty
// barrier), and then releases the next tile's first stage with a row count of -1, which
// stops the MMA warp.
#include "common.cuh"
#include "tcgen05.cuh"
#include "tma_host.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>
#include <stdio.h>

namespace fp4moe {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 192;       // routed rows per tile (MMA N, rounded up to 16 per tile)
constexpr int BK = 64;
// Weight ring: a slot holds 256 k (W_KS k-stages) of a tile's 128 weight rows, so every
// row of the nibble box is one whole 128-byte line and one TMA pair feeds four k-stages.
constexpr int W_KS = 4;
constexpr int W_STAGES = 3;   // weight ring slots (12 k-stages ahead): it streams from HBM
constexpr int A_STAGES = 4;   // converted weight tiles, in tensor memory
// Activation slots of 48 KB: a 192-row tile takes two k-stages per slot (one TMA copy), a
// 32-row tile twelve. On GB300 a CTA completes about one TMA copy per ~270 ns whatever its
// size, so fewer, larger copies pay: three 48 KB slots were 2.9% faster on the prefill
// projections than five 32 KB slots (which, with 192-row tiles at one k-stage per slot,
// had been 6% faster than four); two 72 KB or 64 KB slots were slower.
constexpr int B_STAGES = 3;
constexpr int kMaxExperts = 1024;
// Converter warps per TMEM lane quarter; one of them converts each k-stage of the
// quarter's 32 weight rows, so they take turns over the stages.
constexpr int kConvPerQuarter = 4;
constexpr int kConvTurns = kConvPerQuarter;
constexpr int kConvPerStage = 4;  // one converter warp per TMEM lane quarter per k-stage
constexpr int kThreads = (8 + 4 * kConvPerQuarter) * 32;
// Warp roles. Warp w issues on SM sub-partition w % 4 and reaches TMEM lanes 32 * (w % 4)
// .. + 31 only, so every sub-partition holds one epilogue warp and four converter warps
// for its lane quarter, plus one of: the activation producer (0), the MMA issuer (1), the
// weight producer (2) and the relay (3).
constexpr int kWarpB = 0, kWarpMma = 1, kWarpW = 2, kWarpRelay = 3;
enum { ROLE_RELAY, ROLE_MMA, ROLE_PROD, ROLE_CONV, ROLE_EPI };
__device__ __forceinline__ int warp_role(int w)
{
    if (w == kWarpMma)
        return ROLE_MMA;
    if (w == kWarpB || w == kWarpW)
        return ROLE_PROD;
    if (w == kWarpRelay)
        return ROLE_RELAY;
    return w < 8 ? ROLE_EPI : ROLE_CONV;
}
// Tensor memory (512 columns x 128 lanes of 32 bit): two f32 accumulators of BN columns,
// then the A ring: weight row r in lane r, k-pair j of a stage in column j (16-bit
// elements, even k in the low half), 32 columns per 64-k stage.
constexpr int kACol = 2 * BN;
static_assert(kACol + A_STAGES * (BK / 2) <= 512, "tensor memory budget");
// Activation tiles are loaded k-block-major: one TMA box holds up to 12 k-blocks of a small
// tile (32 rows x 12, 64 x 6, 128 x 3 k-blocks, or BN rows x 2), so small tiles keep many
// k-stages in flight in the same ring slots.
constexpr int B_BYTES = 32 * 12 * BK * 2;  // one ring slot: every box class fills it
constexpr int NIB_BYTES = BM * BK * W_KS / 2;  // 128 rows x 128 bytes, 128-byte swizzle
constexpr int SC_BYTES = BM * 16;               // 16 scale bytes per row (256 k NVFP4)
constexpr int W_BYTES = NIB_BYTES + SC_BYTES;
constexpr int OFF_W = B_STAGES * B_BYTES;
constexpr int RING_BYTES = OFF_W + W_STAGES * W_BYTES;
constexpr int NUM_BARS = 2 * (W_STAGES + A_STAGES + B_STAGES) + 2 + 2 + 1;
// Hardware named barriers (0 is __syncthreads): A slot s is released to the MMA warp
// through barrier kNamedAReady + s, joined by the relay and the MMA warp.
constexpr int kNamedAReady = 1;
constexpr int kNamedThreads = 64;
static_assert(kNamedAReady + A_STAGES <= 16, "named barrier ids");
// Tile row counts the relay publishes to the MMA warp. The relay writes tile i's entry
// after releasing every stage of tiles i - kTileInfo .. i - 1 (at least 2 stages each, as
// k >= 128) and runs at most A_STAGES stages ahead, so with 2 kTileInfo > A_STAGES the
// MMA warp has read the entry's previous tile by then.
constexpr int kTileInfo = A_STAGES;
static_assert(2 * kTileInfo > A_STAGES, "tile info ring depth");
// Tiles looked up ahead for the relay: entry i % kTileRing holds tile i of this CTA (its
// iteration index first, -1 until written), published by the weight producer when it
// starts the tile's copies (at most 16 k-stages, so 4 tiles, ahead of the relay, which
// checks the index before it reads an entry). A lookup (a binary search over the expert
// prefix and two offset reads) cost the relay ~1,000 cycles at every tile start, while the
// MMA warp waited.
constexpr int kTileRing = 16;
constexpr int kTileRingInts = 8;  // seq, e, m, rows, row0 (low, high)
// Epilogue staging (plain output only): each epilogue warp owns a 4 KB buffer, one 32-row
// chunk of its 32 output columns, which one tensor store writes to the output. (Two 2 KB
// halves of 16 rows, one filled while the other's store read it, were ~1 % slower: twice
// the fences, waits and store issues.)
constexpr int kEpiChunkBytes = 32 * 32 * 4;
constexpr int OFF_EPI = (RING_BYTES + NUM_BARS * 8 + 16 + (kMaxExperts + 1) * 4 + kTileInfo * 4 +
                         kTileRing * kTileRingInts * 4 + 1023) & ~1023;
constexpr int SMEM_BYTES = 1024 + OFF_EPI + 4 * kEpiChunkBytes;
static_assert(B_BYTES % 1024 == 0 && W_BYTES % 1024 == 0 && OFF_W % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
static_assert(BN * BK * 2 * 2 <= B_BYTES && BN % 16 == 0 && BN <= 256, "activation box");
static_assert(kThreads <= 1024, "block size");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Params {
    const int32_t *offsets;  // nullable: one expert owning rows [0, P)
    int E;
    int64_t P;
    int n;
    int k;
    int mt;  // weight-row blocks per expert
    const float *scale2;  // nullable: scale2_host is used
    float scale2_host;
    float *out;
    unsigned *err;
    // f16 route (NVFP4): route_flag == 0 after the quantise pass means the workspace holds
    // f16(code * 2^(m - M_p)) and rowscale[p] = 2^M_p; nonzero (or no flag) means bf16.
    const unsigned *route_flag;
    const float *rowscale;
    // bounded-wait limit in clock64 cycles; stall != 0 (a test request) makes the first
    // converter warp of CTA 0 withhold its first arrival, so this launch times out and aborts
    long long wait_limit;
    int stall;
    // nonzero: the output tensor map is valid (row stride a multiple of 16 bytes), and the
    // epilogue writes whole 32-row chunks through it
    int tma_out;
    // fused SwiGLU (gate/up bank: rows [0, inter) gate, [inter, 2 inter) up): out is h
    // [P, inter]; a tile covers 64 h columns (16 gate + 16 up rows per lane quarter)
    int inter;
    float limit;
};

// CSR offset e, or the single-expert offsets {0, P} when the call has none.
__device__ __forceinline__ int64_t offset_at(const Params &p, int e)
{
    return p.offsets ? (int64_t)__ldg(p.offsets + e) : (e == 0 ? 0 : p.P);
}

// ------------------------------------------------------------------ kind::f16 MMA

// One elected lane of a converged warp issues D[tmem] (+)= A[tmem] * B[smem]^T (kind::f16,
// f32 accumulator; a_tmem: lane 0, first column). Operands computed by the whole warp stay
// warp-uniform, which keeps the issue loop short.
__device__ __forceinline__ void mma_f16kind_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem,
                                                        uint64_t b_desc, uint32_t idesc,
                                                        uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "elect.sync r|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Instruction descriptor of kind::f16: f32 accumulator, A and B both bf16 (fmt 1) or both
// f16 (fmt 0), both K-major.
__device__ __forceinline__ uint32_t idesc_f16kind(int m, int n, uint32_t fmt)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h)
{
    const __half2 v = *reinterpret_cast<const __half2 *>(&h);
    return __half22float2(v);
}

// Eight E2M1 nibbles (k order, low nibble first) times a weight scale -> eight bf16,
// exactly (<= 6 significant bits): hardware e2m1x2 -> f16x2 conversion, f32 multiply, bf16
// pack. Measured on this GPU this route converts about 1.65x more weights per cycle than
// a prmt table lookup into bf16 bytes.
__device__ __forceinline__ void e2m1x8_scaled_bf16(uint32_t w, float s, uint4 &out)
{
    uint32_t h[4];
    e2m1x8_to_f16x8(w, h);
    float2 f;
    f = f16x2_to_f32x2(h[0]);
    out.x = pack_bf16x2(f.x * s, f.y * s);
    f = f16x2_to_f32x2(h[1]);
    out.y = pack_bf16x2(f.x * s, f.y * s);
    f = f16x2_to_f32x2(h[2]);
    out.z = pack_bf16x2(f.x * s, f.y * s);
    f = f16x2_to_f32x2(h[3]);
    out.w = pack_bf16x2(f.x * s, f.y * s);
}

// Eight E2M1 nibbles times an e4m3 scale (as f16x2) -> eight f16, exactly: E2M1 x e4m3
// has <= 6 significant bits and lies in [2^-10, 2688], inside f16's normal range.
__device__ __forceinline__ void e2m1x8_scaled_f16(uint32_t w, uint32_t scale_h2, uint4 &out)
{
    uint32_t h[4];
    e2m1x8_to_f16x8(w, h);
    uint32_t *o = &out.x;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[j]) : "r"(h[j]), "r"(scale_h2));
}

// ------------------------------------------------------------------ tile schedule

struct Tile {
    int e;
    int m;
    int64_t row0;
    int rows;
};

__device__ __forceinline__ Tile tile_at(int t, const int *prefix, const Params &p)
{
    const int E = p.E, mt = p.mt;
    int lo = 0, hi = E;  // prefix[lo] <= t < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    Tile tl;
    tl.e = lo;
    const int local = t - prefix[lo];
    const int j = local / mt;
    tl.m = local - j * mt;
    const int64_t r0 = offset_at(p, lo), r1 = offset_at(p, lo + 1);
    tl.row0 = r0 + (int64_t)j * BN;
    const int64_t left = r1 - tl.row0;
    tl.rows = (int)(left < BN ? left : BN);
    return tl;
}

// ------------------------------------------------------------------ the kernel


// Activation tensor maps for tiles of <= 32, 64, 128 and 256 rows: 3-D views {64 k,
// rows, k-blocks} of the [P, k] bf16 workspace with boxes {64, 32 << i, 8 >> i}.
struct BMaps {
    CUtensorMap m[4];
};

__device__ __forceinline__ int bmap_index(int rows)
{
    return rows <= 32 ? 0 : rows <= 64 ? 1 : rows <= 128 ? 2 : 3;
}

// Rows and k-blocks of activation box bi.
__host__ __device__ constexpr int bmap_rows(int bi) { return bi < 3 ? 32 << bi : BN; }
// k-blocks a slot holds: as many as fit in its 32 KB
__host__ __device__ constexpr int bmap_kblocks(int bi)
{
    return bi == 0 ? 12 : bi == 1 ? 6 : bi == 2 ? 3 : 2;
}

// SWIGLU: a weight slot holds eight 16-row blocks (block b: gate rows when b is even, up
// rows when odd, 16 h columns from 64 m + 16 (b / 2)), brought in by one 5-D box
// {k, 16 rows, gate/up, 16-row block, expert} for the nibbles and one for the scales (eight
// 2-D boxes per slot were 4% slower once the stage rate rose), so lane quarter q holds 16
// gate rows in its lanes 0-15 and the matching up rows in lanes 16-31, and the epilogue
// pairs them with one shuffle.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, int c4, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
                 "r"(bar)
                 : "memory");
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ BMaps tmB, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmO,
                   const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + RING_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *prefix = reinterpret_cast<int *>(tmem_slot + 4);
    // tile it's routed-row count (or -1: stop) at tile_info[it % kTileInfo], written by the
    // relay before its first release of the tile's first stage
    volatile int *tile_info = prefix + kMaxExperts + 1;
    volatile int *tile_ring = tile_info + kTileInfo;

    // Values that feed tcgen05 operands are broadcast from lane 0: the compiler then knows
    // they are warp-uniform and issues each tcgen05 instruction once, instead of once per
    // distinct operand value among the lanes.
    const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const uint32_t bar0 = smem_u32(bars);
    // barrier map: weight full/empty, A full/empty, B full/empty, accumulator full/empty, drain
    auto wfull = [&](int s) { return bar0 + 8u * s; };
    auto wempty = [&](int s) { return bar0 + 8u * (W_STAGES + s); };
    auto afull = [&](int s) { return bar0 + 8u * (2 * W_STAGES + s); };
    auto aempty = [&](int s) { return bar0 + 8u * (2 * W_STAGES + A_STAGES + s); };
    auto bfull = [&](int s) { return bar0 + 8u * (2 * W_STAGES + 2 * A_STAGES + s); };
    auto bempty = [&](int s) { return bar0 + 8u * (2 * W_STAGES + 2 * A_STAGES + B_STAGES + s); };
    constexpr int kAcc = 2 * (W_STAGES + A_STAGES + B_STAGES);
    auto accf = [&](int b) { return bar0 + 8u * (kAcc + b); };
    auto acce = [&](int b) { return bar0 + 8u * (kAcc + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (kAcc + 4);

    // --- per-expert tile counts (validated offsets) and their prefix sums
    const int E = p.E;
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const int64_t r0 = offset_at(p, e), r1 = offset_at(p, e + 1);
        const bool bad = r0 < 0 || r1 < r0 || r1 > p.P || (e == 0 && r0 != 0) ||
                         (e == E - 1 && r1 != p.P);
        int cnt = 0;
        if (bad) {
            if (blockIdx.x == 0)
                raise_device_error(p.err, FP4_DEVERR_OFFSETS);
        } else if (r1 > r0) {
            cnt = (int)((r1 - r0 + BN - 1) / BN) * p.mt;
        }
        prefix[e + 1] = cnt;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < W_STAGES; ++s) {
            mbar_init(wfull(s), 1);
            mbar_init(wempty(s), kConvPerStage * W_KS);
        }
        for (int s = 0; s < A_STAGES; ++s) {
            mbar_init(afull(s), kConvPerStage);
            mbar_init(aempty(s), 1);
        }
        for (int s = 0; s < B_STAGES; ++s) {
            mbar_init(bfull(s), 1);
            mbar_init(bempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf(b), 1);
            mbar_init(acce(b), 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        prefix[0] = 0;
        for (int i = 0; i < kTileRing; ++i)
            tile_ring[i * kTileRingInts] = -1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpMma)
        tmem_alloc(smem_u32(tmem_slot), 512);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = __shfl_sync(0xFFFFFFFFu, *tmem_slot, 0);
    const int total = prefix[E];
    const bool f16_route = p.route_flag != nullptr && *((volatile const unsigned *)p.route_flag) == 0u;
    const int nkb = p.k / BK;
    uint8_t *const ringB = smem;
    uint8_t *const ringW = smem + OFF_W;

    const int role = warp_role(warp);
    if (role == ROLE_PROD) {
        // ---------------------------------------------------------- TMA producers
        // kWarpB: activation slots into the B ring; kWarpW: nibbles + scales into the W ring
        if (lane == 0) {
            const bool is_b = warp == kWarpB;
            const int nslots = is_b ? B_STAGES : W_STAGES;
            int slot = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int t = blockIdx.x, pit = 0; t < total && ok; t += gridDim.x, ++pit) {
                const Tile tl = tile_at(t, prefix, p);
                if (!is_b) {  // publish the lookup for the relay (entry pit % kTileRing)
                    volatile int *ent = tile_ring + (pit % kTileRing) * kTileRingInts;
                    ent[1] = tl.e;
                    ent[2] = tl.m;
                    ent[3] = tl.rows;
                    ent[4] = (int)(uint32_t)((uint64_t)tl.row0 & 0xFFFFFFFFu);
                    ent[5] = (int)(uint32_t)((uint64_t)tl.row0 >> 32);
                    __threadfence_block();
                    ent[0] = pit;
                }
                const int yw = tl.e * p.n + tl.m * BM;
                const int bi = bmap_index(tl.rows);
                const int kbps = bmap_kblocks(bi);
                const uint32_t box_bytes = (uint32_t)(bmap_rows(bi) * kbps * BK * 2);
                const int nload = is_b ? (nkb + kbps - 1) / kbps : nkb / W_KS;
                for (int j = 0; j < nload; ++j) {
                    const uint32_t emp = is_b ? bempty(slot) : wempty(slot);
                    const uint32_t ful = is_b ? bfull(slot) : wfull(slot);
                    if (!mbar_wait(emp, phase ^ 1u, abort_flag, p.err, p.wait_limit)) {
                        ok = false;
                        break;
                    }
                    if (is_b) {
                        mbar_arrive_expect_tx(ful, box_bytes);
                        tma_load_3d(smem_u32(ringB + slot * B_BYTES), &tmB.m[bi], 0, (int)tl.row0,
                                    j * kbps, ful);
                    } else {
                        uint8_t *dst = ringW + slot * W_BYTES;
                        const int k0 = j * W_KS * BK;  // first k of the slot
                        mbar_arrive_expect_tx(ful, W_BYTES);
                        if (SWIGLU) {
                            // one 5-D box each: {k, row of a 16-row block, gate/up, block, expert}
                            tma_load_5d(smem_u32(dst), &tmW, k0 / 2, 0, 0, tl.m * 4, tl.e, ful);
                            tma_load_5d(smem_u32(dst + NIB_BYTES), &tmS, k0 / 16, 0, 0, tl.m * 4, tl.e,
                                        ful);
                        } else {
                            tma_load_2d(smem_u32(dst), &tmW, k0 / 2, yw, ful);
                            tma_load_2d(smem_u32(dst + NIB_BYTES), &tmS, k0 / 16, yw, ful);
                        }
                    }
                    issued_mask |= 1u << slot;
                    issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
                    if (++slot == nslots) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {  // let this CTA's own copies land before it exits
                for (int s = 0; s < nslots; ++s)
                    if (issued_mask & (1u << s))
                        mbar_drain(is_b ? bfull(s) : wfull(s), (issued_parity >> s) & 1u);
            }
        }
    } else if (role == ROLE_MMA) {
        // ---------------------------------------------------------- MMA issuer
        // The whole warp runs the loop; one elected lane issues each MMA and commit. It never
        // waits on an mbarrier, and it reads shared memory once per tile (the row count the
        // relay published), right after the tile's first named barrier (see the header).
        unsigned st = 0;  // A stages issued (A slot = st % A_STAGES, the relay's order)
        int bslot = 0;  // activation ring slot
        int it = 0;
        // B descriptor of ring slot 0; other slots and k-blocks only move the start address
        const uint64_t bdesc0 = sw128_desc(smem_u32(ringB));
        const uint32_t a_tmem0 = tmem_base + (uint32_t)kACol;
        const uint32_t ab_fmt = __shfl_sync(0xFFFFFFFFu, f16_route ? 0u : 1u, 0);
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            named_sync(kNamedAReady + (int)(st % A_STAGES), kNamedThreads);  // tile's first stage
            const int rows = __shfl_sync(0xFFFFFFFFu, tile_info[it % kTileInfo], 0);
            if (rows < 0)
                break;  // the relay is aborting
            const int nt = max(16, (rows + 15) & ~15);
            const uint32_t idesc = idesc_f16kind(BM, nt, ab_fmt);
            const int buf = it & 1;
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
            const int bi = bmap_index(rows);
            const int kbps = bmap_kblocks(bi);
            const uint32_t kb_desc = (uint32_t)(bmap_rows(bi) * BK * 2) >> 4;  // one k-block
            int j = 0;  // k-block of the current activation slot
            // one k-stage; the relay has seen: accumulator free (kb 0), activation slot full
            // (j 0), converted weight slot full
            auto stage = [&](int kb) {
                const int as = (int)(st % A_STAGES);
                tc_fence_after();
                const uint32_t a_tmem = a_tmem0 + (uint32_t)(as * (BK / 2));
                const uint64_t bdesc =
                    bdesc0 + (uint64_t)(bslot * (B_BYTES >> 4) + (uint32_t)j * kb_desc);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_f16kind_tmem_a_warp(d_tmem, a_tmem + 8u * kk, bdesc + 2u * kk, idesc,
                                            (kb | kk) != 0 ? 1u : 0u);
                mma_commit_warp(aempty(as));
                ++st;
                if (j == kbps - 1 || kb == nkb - 1) {
                    mma_commit_warp(bempty(bslot));
                    bslot = bslot + 1 == B_STAGES ? 0 : bslot + 1;
                    j = 0;
                } else {
                    ++j;
                }
            };
            stage(0);
            for (int kb = 1; kb < nkb; ++kb) {
                named_sync(kNamedAReady + (int)(st % A_STAGES), kNamedThreads);
                stage(kb);
            }
            mma_commit_warp(accf(buf));
        }
        mma_commit_warp(drain_bar);  // completes once every MMA issued above has finished
        warp_mbar_drain(drain_bar, 0);
    } else if (role == ROLE_RELAY) {
        // ---------------------------------------------------------- relay
        // Walks the MMA warp's stage sequence, waits for what each stage needs and
        // releases its A slot with bar.arrive. A slot's next use is full only after the
        // converters saw the MMAs of its previous use complete, so the relay can never
        // lap the MMA warp on a named barrier.
        // The converters run ahead of the MMAs, and an mbarrier wait costs this warp a
        // few hundred cycles even on a completed phase (its SM sub-partition is busy with
        // converter work), which made the relay the pace-setter at small N. So lanes 0-3
        // test the A slots of the next four stages in one instruction, and the stages
        // found full are released without another wait.
        Ring<A_STAGES> ra;
        Ring<B_STAGES> rb;
        int it = 0;
        int a_ready = 0;  // stages from ra on whose converted A slot is known to be full
        bool aborted = false, stuck = false;
        for (int t = blockIdx.x; t < total && !aborted; t += gridDim.x, ++it) {
            Tile tl;
            volatile int *ent = tile_ring + (it % kTileRing) * kTileRingInts;
            if (ent[0] == it) {  // looked up ahead by the epilogue
                __threadfence_block();
                tl.e = ent[1];
                tl.m = ent[2];
                tl.rows = ent[3];
                tl.row0 = (int64_t)(((uint64_t)(uint32_t)ent[5] << 32) | (uint32_t)ent[4]);
            } else {
                tl = tile_at(t, prefix, p);
            }
            const int buf = it & 1;
            // published before the arrival that releases the tile's first stage
            tile_info[it % kTileInfo] = tl.rows;
            bool ok = warp_mbar_wait(acce(buf), ((it >> 1) & 1) ^ 1u, abort_flag, p.err, p.wait_limit);
            const int kbps = bmap_kblocks(bmap_index(tl.rows));
            int j = 0;  // k-block of the current activation slot
            for (int kb = 0; kb < nkb; ++kb) {
                if (ok && j == 0)
                    ok = warp_mbar_wait(bfull(rb.slot), rb.phase, abort_flag, p.err, p.wait_limit);
                if (ok && a_ready == 0) {
                    // stage l ahead uses slot ra.slot + l (mod A_STAGES), one phase later
                    // if that wraps; its previous use was released already, so a full
                    // phase of that parity is this stage's
                    bool full_l = false;
                    if (lane < A_STAGES) {
                        const int sl = ra.slot + lane;
                        full_l = mbar_test(afull(sl % A_STAGES), ra.phase ^ (sl >= A_STAGES ? 1u : 0u));
                    }
                    const unsigned full_m = __ballot_sync(0xFFFFFFFFu, full_l);
                    __syncwarp();
                    a_ready = __ffs(~full_m) - 1;  // consecutive full stages from ra
                    if (a_ready == 0) {
                        ok = warp_mbar_wait(afull(ra.slot), ra.phase, abort_flag, p.err, p.wait_limit);
                        a_ready = 1;
                    }
                }
                if (!ok) {
                    // Aborting: keep the MMA warp moving to the end of this tile, then stop
                    // it at the next tile start. Release a slot only after the MMAs of its
                    // previous use completed, so that no barrier generation pairs two
                    // arrivals of the relay.
                    aborted = true;
                    if (!warp_mbar_drain(aempty(ra.slot), ra.phase ^ 1u)) {
                        stuck = true;
                        break;
                    }
                }
                named_arrive(kNamedAReady + ra.slot, kNamedThreads);
                ra.next();
                a_ready = a_ready > 0 ? a_ready - 1 : 0;
                if (j == kbps - 1 || kb == nkb - 1) {
                    rb.next();
                    j = 0;
                } else {
                    ++j;
                }
            }
            if (stuck)
                break;
            if (aborted && t + (int)gridDim.x < total) {
                // the MMA warp would start another tile: release its first stage with a
                // row count of -1, which makes it stop
                tile_info[(it + 1) % kTileInfo] = -1;
                if (warp_mbar_drain(aempty(ra.slot), ra.phase ^ 1u))
                    named_arrive(kNamedAReady + ra.slot, kNamedThreads);
            }
        }
    } else if (role == ROLE_CONV) {
        // ---------------------------------------------------------- converters
        // Warp w writes TMEM lane quarter q = w % 4 (the only lanes its tcgen05.st reaches):
        // lane i converts weight row 32 q + i. The four converter warps of a quarter take
        // turns over the k-stages (h = 0 .. 3 converts stages h, h + 4, ...), each the whole
        // 64-k stage of its rows: two 16-byte nibble chunks, one 32-column tensor-memory store.
        const int q = warp & 3, h = (warp - 8) >> 2;
        const int r = q * 32 + lane;
        const uint32_t a_lane = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)kACol;
        const int ntiles = (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        const int nst = ntiles * nkb;
        // g: this CTA's k-stage sequence over its tiles. Every tile has a multiple of W_KS
        // stages, so W slot g / W_KS holds stage g as its sub-stage g % W_KS; kConvTurns is a
        // multiple of W_KS, so this warp always takes the same sub-stage of a slot.
        static_assert(kConvTurns % W_KS == 0 && kConvTurns % A_STAGES == 0, "converter turns");
        const int sub = h % W_KS, aslot = h % A_STAGES;
        const uint8_t *const nib_row = ringW + r * 128;
        const int off0 = ((2 * sub) ^ (r & 7)) << 4, off1 = ((2 * sub + 1) ^ (r & 7)) << 4;
        int wslot = 0;
        uint32_t wphase = 0, aphase = 0;
        for (int g = h; g < nst; g += kConvTurns) {
            if (!mbar_wait(wfull(wslot), wphase, abort_flag, p.err, p.wait_limit))
                break;
            const uint8_t *w = ringW + wslot * W_BYTES;
            // row r of the nibble box is 128 bytes in the 128-byte swizzle: its 16-byte chunk
            // j (32 k) sits at chunk j ^ (r & 7); a warp's 32 rows then read conflict-free
            const uint4 n0 = *reinterpret_cast<const uint4 *>(nib_row + wslot * W_BYTES + off0);
            const uint4 n1 = *reinterpret_cast<const uint4 *>(nib_row + wslot * W_BYTES + off1);
            uint32_t o[32];
            uint4 *o4 = reinterpret_cast<uint4 *>(o);
            // the slot's 16 scale bytes of row r cover its 256 k; this stage's four are word sub
            {
                const uint32_t s4 = *reinterpret_cast<const uint32_t *>(w + NIB_BYTES + r * 16 + 4 * sub);
                if (f16_route) {
                    const uint32_t h0 = e4m3x2_to_f16x2((s4 & 0xFFu) * 0x101u);
                    const uint32_t h1 = e4m3x2_to_f16x2(((s4 >> 8) & 0xFFu) * 0x101u);
                    const uint32_t h2 = e4m3x2_to_f16x2(((s4 >> 16) & 0xFFu) * 0x101u);
                    const uint32_t h3 = e4m3x2_to_f16x2((s4 >> 24) * 0x101u);
                    e2m1x8_scaled_f16(n0.x, h0, o4[0]);
                    e2m1x8_scaled_f16(n0.y, h0, o4[1]);
                    e2m1x8_scaled_f16(n0.z, h1, o4[2]);
                    e2m1x8_scaled_f16(n0.w, h1, o4[3]);
                    e2m1x8_scaled_f16(n1.x, h2, o4[4]);
                    e2m1x8_scaled_f16(n1.y, h2, o4[5]);
                    e2m1x8_scaled_f16(n1.z, h3, o4[6]);
                    e2m1x8_scaled_f16(n1.w, h3, o4[7]);
                } else {
                    const float f0 = e4m3_to_f32(s4 & 0xFFu), f1 = e4m3_to_f32((s4 >> 8) & 0xFFu);
                    const float f2 = e4m3_to_f32((s4 >> 16) & 0xFFu), f3 = e4m3_to_f32(s4 >> 24);
                    e2m1x8_scaled_bf16(n0.x, f0, o4[0]);
                    e2m1x8_scaled_bf16(n0.y, f0, o4[1]);
                    e2m1x8_scaled_bf16(n0.z, f1, o4[2]);
                    e2m1x8_scaled_bf16(n0.w, f1, o4[3]);
                    e2m1x8_scaled_bf16(n1.x, f2, o4[4]);
                    e2m1x8_scaled_bf16(n1.y, f2, o4[5]);
                    e2m1x8_scaled_bf16(n1.z, f3, o4[6]);
                    e2m1x8_scaled_bf16(n1.w, f3, o4[7]);
                }
            }
            // Release the weight slot once its values are consumed, behind an async-proxy
            // fence that orders these reads before the TMA refill. (Arriving right after
            // issuing the reads let the refill land first: wrong weight rows on GB300.)
            fence_proxy_async();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(wempty(wslot));
            // then wait for the A slot: the conversion overlapped the MMAs still reading it
            if (!mbar_wait(aempty(aslot), aphase ^ 1u, abort_flag, p.err, p.wait_limit))
                break;
            tc_fence_after();
            tmem_st32(a_lane + (uint32_t)(aslot * (BK / 2)), o);
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && !(p.stall && blockIdx.x == 0 && warp == 8 && g == h))
                mbar_arrive(afull(aslot));
            // next stage g + kConvTurns: W slot sequence + kConvTurns / W_KS, A slot the same
            // (kConvTurns is a multiple of A_STAGES), the A phase flips every kConvTurns /
            // A_STAGES uses
            for (int i = 0; i < kConvTurns / W_KS; ++i)
                if (++wslot == W_STAGES) {
                    wslot = 0;
                    wphase ^= 1u;
                }
            aphase ^= (uint32_t)((kConvTurns / A_STAGES) & 1);
        }
    } else if (role == ROLE_EPI) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        float *stg = reinterpret_cast<float *>(smem + OFF_EPI + q * kEpiChunkBytes);
        const uint32_t stg_s = smem_u32(stg);
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const Tile tl = tile_at(t, prefix, p);
            const int buf = it & 1;
            // The tile's global reads (its routed rows' scales, lane j holding row 32 c + j,
            // and scale2) are issued before the wait for the accumulator: read chunk by chunk
            // after it, each waited behind the kernel's own copies, and the accumulator's
            // release for tile it + 2 came ~2,000 (N = 64) to ~6,400 (N = 192) cycles late.
            float rsv[BN / 32];
#pragma unroll
            for (int cc = 0; cc < BN / 32; ++cc) {
                const int rr = cc * 32 + lane;
                rsv[cc] = f16_route && rr < tl.rows ? __ldg(p.rowscale + tl.row0 + rr) : 1.0f;
            }
            const float s2 = p.scale2 ? __ldg(p.scale2 + tl.e) : p.scale2_host;
            if (!mbar_wait(accf(buf), (it >> 1) & 1, abort_flag, p.err, p.wait_limit))
                break;
            tc_fence_after();
            // SWIGLU: TMEM lanes 0-15 of the quarter hold gate rows and 16-31 the matching up
            // rows; h column col is computed by lane col % 16 for even routed rows and by
            // lane 16 + col % 16 for odd ones
            const int col0 = SWIGLU ? tl.m * 64 + q * 16 : tl.m * BM + q * 32;
            const int col = col0 + (SWIGLU ? (lane & 15) : lane);
            const int ldo = SWIGLU ? p.inter : p.n;
            const bool colok = SWIGLU ? col < p.inter : col < p.n;
            float *orow = p.out + tl.row0 * (int64_t)ldo + col;
#pragma unroll
            for (int cc = 0; cc < BN / 32; ++cc) {
                const int c0 = cc * 32;
                if (c0 >= tl.rows)
                    break;
                uint32_t v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c0), v);
                // f16 route: column (routed row) scale 2^M_p, exact; lane j holds row c0 + j
                const float rs = rsv[cc];
                if (!SWIGLU && p.tma_out && c0 + 32 <= tl.rows && col0 < ldo) {
                    // A whole chunk leaves through shared memory and one tensor store: a
                    // shared store per value has no address arithmetic and no wait on the
                    // global store path, which made the epilogue of a 192-row tile release
                    // its accumulator late. Columns past the output's width are cut off by
                    // the tensor store. (Under SwiGLU, with 64-byte h rows per warp, staged
                    // stores made the fused gate/up call slower instead.)
                    if (lane == 0)
                        bulk_wait_read_all();  // the previous chunk's store has read the buffer
                    __syncwarp();
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const float r = f16_route ? __shfl_sync(0xFFFFFFFFu, rs, jj) : 1.0f;
                        stg[jj * 32 + lane] = (__uint_as_float(v[jj]) * r) * s2;
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmO, stg_s, col0, (int)(tl.row0 + c0));
                        bulk_commit();
                    }
                } else if constexpr (SWIGLU) {
                    // two routed rows a step: lanes 0-15 take row jj (gate here, up from lane
                    // + 16), lanes 16-31 row jj + 1 (gate from lane - 16, up here), so each
                    // lane evaluates SwiGLU once per two rows and a store covers both rows
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 2) {
                        // f16_route is uniform over the CTA, so every lane takes the shuffles
                        const float ra = f16_route ? __shfl_sync(0xFFFFFFFFu, rs, jj) : 1.0f;
                        const float rb = f16_route ? __shfl_sync(0xFFFFFFFFu, rs, jj + 1) : 1.0f;
                        const float va = (__uint_as_float(v[jj]) * ra) * s2;
                        const float vb = (__uint_as_float(v[jj + 1]) * rb) * s2;
                        const float other = __shfl_xor_sync(0xFFFFFFFFu, lane < 16 ? vb : va, 16);
                        const float gate = lane < 16 ? va : other, up = lane < 16 ? other : vb;
                        const int row = c0 + jj + (lane >> 4);
                        if (colok && row < tl.rows)
                            orow[(int64_t)row * ldo] = swiglu_one(gate, up, p.limit);
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        // f16_route is uniform over the CTA, so every lane takes the shuffle
                        const float r = f16_route ? __shfl_sync(0xFFFFFFFFu, rs, jj) : 1.0f;
                        if (colok && c0 + jj < tl.rows)
                            orow[(int64_t)(c0 + jj) * ldo] = (__uint_as_float(v[jj]) * r) * s2;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce(buf));
        }
        if (lane == 0)
            bulk_wait_all();  // the staged halves stay in use until their stores complete
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------ quantise pass

// Largest exponent gap between a row's block scales that f16 still holds exactly: codes
// are multiples of 2^-9, so code * 2^-15 is a multiple of 2^-24, f16's finest spacing.
constexpr int kF16MaxScaleGap = 15;
// 128-groups a warp of the quantise pass holds in registers (rows up to k = 8 * 8 * 128).
constexpr int kQuantRegGroups = 8;

// act_quant of one 128-group held as a float4 per lane (fn quant_rows of
// dsv4_native_gemm_gate.rs): returns the group scale 2^m (shuffle max, floor 1e-4, times
// f32(1/448), pow2_ceil) and this lane's four e4m3 codes, packed.
__device__ __forceinline__ float quant_group4(const float4 v, uint32_t &q)
{
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = warp_max(amax);
    const float s = group_scale(amax);
    const float inv = pow2_reciprocal(s);
    q = e4m3x4(scaled_clamped(v.x, inv), scaled_clamped(v.y, inv), scaled_clamped(v.z, inv),
               scaled_clamped(v.w, inv));
    return s;
}

// The 16-bit MMA operands of four packed codes: f16(code * mul) with mul = 2^(m - M) in
// [2^-15, 1] (f16 route), or bf16(code * 2^m) (bf16 route). Both exact.
__device__ __forceinline__ uint2 ws_word(uint32_t q, float mul, bool f16)
{
    const float2 lo = f16x2_to_f32x2(e4m3x2_to_f16x2(q & 0xFFFFu));
    const float2 hi = f16x2_to_f32x2(e4m3x2_to_f16x2(q >> 16));
    uint2 o;
    if (f16) {
        o.x = pack_f16x2(lo.x * mul, lo.y * mul);
        o.y = pack_f16x2(hi.x * mul, hi.y * mul);
    } else {
        o.x = pack_bf16x2(lo.x * mul, lo.y * mul);
        o.y = pack_bf16x2(hi.x * mul, hi.y * mul);
    }
    return o;
}

// Quantise pass: routed row p of the workspace = the 16-bit MMA operand of act_quant of
// activation row x[row_ids[p]] (x[p] without row ids), in one of two forms:
//   f16 route (NVFP4): f16(code * 2^(m_b - M_p)) and rowscale[p] = 2^M_p, M_p the row's
//       largest block exponent; exact while every block lies within 2^15 of M_p. A row
//       with a wider spread sets *route_flag and is not written: the bf16 pass then
//       rewrites every row (the GEMM takes one operand type per call).
//   bf16 route (the f16 route's fallback): bf16(code * 2^m_b), always exact.
// A CTA of 8 warps takes 8 / wr rows at a time; the wr warps of a row split its 128-groups
// (warp i of the row takes groups i, i + wr, ...). With REG (at most kQuantRegGroups
// groups per warp) the row stays in registers between the scale reduction and the
// writes, so it is read once; otherwise (k above 8192) the f16 route reads it twice.
// Rows whose id is outside [0, T) are written as zeros and raise FP4_DEVERR_ROW_ID.
// With only_if set, the kernel runs only when *only_if is nonzero.
template <bool REG>
__global__ void __launch_bounds__(256, 3) quant_ws_kernel(const float *__restrict__ x, int64_t T,
                                                       const int32_t *__restrict__ row_ids,
                                                       int64_t P, int k, int wr, int f16_route,
                                                       uint2 *__restrict__ ws,
                                                       float *__restrict__ rowscale,
                                                       unsigned *route_flag,
                                                       const unsigned *only_if, unsigned *err)
{
    if (only_if && *((volatile const unsigned *)only_if) == 0u)
        return;
    __shared__ uint32_t red[2][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kq = k >> 7;
    const int rpc = 8 / wr;
    const int slot = warp / wr, wi = warp - slot * wr;
    const bool f16 = f16_route != 0;
    for (int64_t base = (int64_t)blockIdx.x * rpc; base < P; base += (int64_t)gridDim.x * rpc) {
        const int64_t pr = base + slot;
        const bool have = pr < P;
        const int64_t t = have ? (row_ids ? (int64_t)__ldg(row_ids + pr) : pr) : -1;
        const bool valid = t >= 0 && t < T;
        if (have && !valid && wi == 0 && lane == 0)
            raise_device_error(err, FP4_DEVERR_ROW_ID);
        const float4 *xr = reinterpret_cast<const float4 *>(x + (valid ? t : 0) * (int64_t)k);
        uint2 *wrow = ws + pr * (int64_t)(k / 4);
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
        uint32_t emax = 0u, emin = 255u;
        uint32_t c[kQuantRegGroups];
        float s[kQuantRegGroups];
        if (REG) {
            float4 v[kQuantRegGroups];
#pragma unroll
            for (int i = 0; i < kQuantRegGroups; ++i) {
                const int g = wi + i * wr;
                v[i] = (valid && g < kq) ? __ldg(xr + g * 32 + lane) : zero;
            }
#pragma unroll
            for (int i = 0; i < kQuantRegGroups; ++i) {
                if (wi + i * wr < kq) {  // uniform over the warp
                    s[i] = quant_group4(v[i], c[i]);
                    const uint32_t e = __float_as_uint(s[i]) >> 23;
                    emax = max(emax, e);
                    emin = min(emin, e);
                }
            }
        } else if (f16) {
            for (int g = wi; g < kq; g += wr) {
                uint32_t cc;
                const uint32_t e =
                    __float_as_uint(quant_group4(valid ? __ldg(xr + g * 32 + lane) : zero, cc)) >> 23;
                emax = max(emax, e);
                emin = min(emin, e);
            }
        }
        if (f16) {  // the row's largest and smallest block exponent, over its wr warps
            if (lane == 0) {
                red[0][warp] = emax;
                red[1][warp] = emin;
            }
            __syncthreads();
            for (int j = 0; j < wr; ++j) {
                emax = max(emax, red[0][slot * wr + j]);
                emin = min(emin, red[1][slot * wr + j]);
            }
        }
        const bool wide = f16 && emin + kF16MaxScaleGap < emax;
        if (have && wide && wi == 0 && lane == 0)
            atomicOr(route_flag, 1u);
        if (have && !wide) {
            if (f16 && wi == 0 && lane == 0)
                rowscale[pr] = __uint_as_float(emax << 23);
            if (REG) {
#pragma unroll
                for (int i = 0; i < kQuantRegGroups; ++i) {
                    const int g = wi + i * wr;
                    if (g < kq) {
                        // 2^(m - M) in [2^-15, 1] (f16 route), or the group scale (bf16)
                        const float mul =
                            f16 ? __uint_as_float(((__float_as_uint(s[i]) >> 23) + 127u - emax) << 23)
                                : s[i];
                        wrow[g * 32 + lane] = ws_word(c[i], mul, f16);
                    }
                }
            } else {
                for (int g = wi; g < kq; g += wr) {
                    uint32_t cc;
                    const float sg = quant_group4(valid ? __ldg(xr + g * 32 + lane) : zero, cc);
                    const float mul =
                        f16 ? __uint_as_float(((__float_as_uint(sg) >> 23) + 127u - emax) << 23) : sg;
                    wrow[g * 32 + lane] = ws_word(cc, mul, f16);
                }
            }
        }
        if (f16)
            __syncthreads();  // red[] is rewritten by the next rows
    }
}

// Expand: routed row p of the GEMM's workspace = token row row_ids[p] of the per-token
// workspace (its 16-bit operands and, on the f16 route, its row scale), a copy. One warp
// per routed row; 16-byte loads kept in L2 (the token rows are read about topk times),
// streaming stores. Row ids outside [0, T) give zero rows and raise FP4_DEVERR_ROW_ID.
__global__ void __launch_bounds__(256) expand_ws_kernel(const uint4 *__restrict__ tok_act,
                                                        const float *__restrict__ tok_scale,
                                                        const int32_t *__restrict__ row_ids,
                                                        int64_t T, int64_t P, int k,
                                                        uint4 *__restrict__ act,
                                                        float *__restrict__ rowscale,
                                                        unsigned *err)
{
    const int lane = threadIdx.x & 31;
    const int chunks = k / 8;  // 16-byte chunks of a row of k 16-bit values
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t pr = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pr < P;
         pr += warps) {
        const int64_t t = __ldg(row_ids + pr);
        const bool ok = t >= 0 && t < T;
        if (!ok && lane == 0)
            raise_device_error(err, FP4_DEVERR_ROW_ID);
        const uint4 *src = tok_act + (ok ? t : 0) * chunks;
        uint4 *dst = act + pr * chunks;
        for (int c = lane; c < chunks; c += 32) {
            const uint4 v = ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            __stcs(dst + c, v);
        }
        if (lane == 0)
            rowscale[pr] = ok ? __ldg(tok_scale + t) : 1.0f;
    }
}

// 3-D map {64 k, rows, k-blocks} over a [rows, k] bf16 matrix, box {64, box_rows, box_kb}.
static bool make_map_kblocks(CUtensorMap *m, const void *base, uint64_t k, uint64_t rows,
                             uint32_t box_rows, uint32_t box_kb)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)BK, rows, k / BK};
    cuuint64_t strides[2] = {k * 2, (cuuint64_t)BK * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, box_kb};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

} // namespace tc

// Tokens are quantised once when routed rows repeat them (row ids given and fewer tokens
// than routed rows): into a per-token region, then copied into routed-row order; otherwise
// the quantise pass reads every routed row's activation directly.
static bool per_token(const GroupedProblem &p)
{
    return p.row_ids != nullptr && p.T < p.P;
}

static size_t ws_act_bytes(int64_t rows, int64_t k)
{
    return ((size_t)rows * (size_t)k * 2 + 1023) & ~(size_t)1023;
}

static size_t ws_rows_bytes(int64_t rows, int64_t k)
{
    return ws_act_bytes(rows, k) + (((size_t)rows * 4 + 1023) & ~(size_t)1023);
}

// Workspace: [routed rows: P x k 16-bit operands | P row scales][route flag, 1 KB]
// [when tokens repeat: T x k 16-bit operands | T row scales], each part 1024-aligned.
size_t tc_workspace_bytes(int64_t num_tokens, int64_t total_rows, int64_t k, int recipe)
{
    (void)recipe;
    size_t b = 1024 + ws_rows_bytes(total_rows, k) + 1024;
    if (num_tokens < total_rows)
        b += ws_rows_bytes(num_tokens, k);
    return b;
}

bool tc_supported(int64_t n, int64_t k, int recipe, int E)
{
    const int gs = recipe == FP4_NVFP4 ? 16 : 32;
    if (k % (16 * gs) != 0 || k % tc::BK != 0)
        return false;  // the scale tensor's rows must be whole 16-byte TMA units
    if (E < 1 || E > tc::kMaxExperts || (int64_t)E * n >= ((int64_t)1 << 31))
        return false;
    return n >= 1;
}

// Multiprocessor count of the current device, looked up once per device.
static int device_sms()
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

// Where the parts of a workspace live.
struct WsLayout {
    uint8_t *act;          // [P, k] 16-bit MMA operands in routed-row order
    float *rowscale;       // [P] f32 (f16 route)
    unsigned *route_flag;  // nonzero: the bf16 route holds
    uint8_t *tok_act;      // [T, k] per token (when tokens repeat)
    float *tok_scale;      // [T]
};

static WsLayout ws_layout(const void *workspace, int64_t T, int64_t P, int64_t k)
{
    WsLayout l;
    l.act = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(workspace) + 1023) &
                                        ~(uintptr_t)1023);
    l.rowscale = reinterpret_cast<float *>(l.act + ws_act_bytes(P, k));
    l.route_flag = reinterpret_cast<unsigned *>(l.act + ws_rows_bytes(P, k));
    l.tok_act = l.act + ws_rows_bytes(P, k) + 1024;
    l.tok_scale = reinterpret_cast<float *>(l.tok_act + ws_act_bytes(T, k));
    return l;
}

// Quantise pass of the NVFP4 tensor-core path: every routed row into the workspace. It
// first tries f16 with a per-row power-of-two scale (the cheaper weight conversion in the
// GEMM); if any row's block scales span more than f16 holds exactly, the bf16 pass rewrites
// all rows. (MXFP4 has its own pass and kernel: the block-scaled 8-bit MMA.)
cudaError_t launch_tc_quantize(const GroupedProblem &p, void *workspace, cudaStream_t s)
{
    using namespace tc;
    if (p.recipe != FP4_NVFP4)
        return cudaErrorInvalidValue;
    const bool tok = per_token(p);
    const WsLayout l = ws_layout(workspace, p.T, p.P, p.k);
    const int64_t S = tok ? p.T : p.P;                 // rows the quantise pass writes
    const int32_t *rid = tok ? nullptr : p.row_ids;    // per token: row s is x[s]
    uint2 *qact = reinterpret_cast<uint2 *>(tok ? l.tok_act : l.act);
    float *qscale = tok ? l.tok_scale : l.rowscale;
    const int sms = device_sms();
    const int kq = p.k / 128;
    // warps per row: enough that each holds at most kQuantRegGroups groups, a power of two <= 8
    int wr = 1;
    while (wr < 8 && (kq + wr - 1) / wr > kQuantRegGroups)
        wr <<= 1;
    const bool reg = (kq + wr - 1) / wr <= kQuantRegGroups;
    const int64_t rpc = 8 / wr;
    const int64_t want = (S + rpc - 1) / rpc;
    const int blocks = (int)(want < (int64_t)sms * 3 ? want : (int64_t)sms * 3);  // 3 CTAs per SM
    auto kern = reg ? quant_ws_kernel<true> : quant_ws_kernel<false>;
    cudaError_t e = cudaMemsetAsync(l.route_flag, 0, sizeof(unsigned), s);
    if (e != cudaSuccess)
        return e;
    if (S > 0) {
        kern<<<blocks, 256, 0, s>>>(p.x, p.T, rid, S, p.k, wr, 1, qact, qscale, l.route_flag,
                                    nullptr, p.err);
        // the bf16 fallback: exits at once unless a row was too wide for f16 (the host cannot
        // know without a synchronisation, so it is always enqueued)
        const int fb = 2 * sms < blocks ? 2 * sms : blocks;
        kern<<<fb, 256, 0, s>>>(p.x, p.T, rid, S, p.k, wr, 0, qact, qscale, nullptr,
                                l.route_flag, p.err);
    }
    if (tok) {
        const int64_t ew = (p.P + 7) / 8;
        const int eblocks = (int)(ew < (int64_t)sms * 8 ? ew : (int64_t)sms * 8);
        expand_ws_kernel<<<eblocks, 256, 0, s>>>(
            reinterpret_cast<const uint4 *>(l.tok_act), l.tok_scale, p.row_ids, p.T, p.P, p.k,
            reinterpret_cast<uint4 *>(l.act), l.rowscale, p.err);
    }
    return cudaGetLastError();
}

// The persistent NVFP4 tensor-core GEMM over a workspace that launch_tc_quantize filled
// for the same tokens, row ids (present or not), routed rows and k. With sw, the bank is a
// gate/up bank of n = 2 inter rows and the epilogue writes h = SwiGLU(gate, up) [P, inter].
cudaError_t launch_tc_gemm(const GroupedProblem &p, const void *workspace, cudaStream_t s,
                           const SwigluOut *sw)
{
    using namespace tc;
    if (p.recipe != FP4_NVFP4 || !tc_supported(p.n, p.k, p.recipe, p.E))
        return cudaErrorInvalidValue;
    if (sw && (sw->inter % 64 != 0 || 2 * sw->inter != p.n))
        return cudaErrorInvalidValue;
    const WsLayout l = ws_layout(workspace, p.T, p.P, p.k);
    const int sms = device_sms();
    const uint32_t wbox = sw ? 16 : BM;  // rows per weight box
    alignas(64) BMaps tmB;
    alignas(64) CUtensorMap tmW, tmS;
    for (int i = 0; i < 4; ++i)
        if (!make_map_kblocks(&tmB.m[i], l.act, (uint64_t)p.k, (uint64_t)p.P,
                              (uint32_t)bmap_rows(i), (uint32_t)bmap_kblocks(i)))
            return cudaErrorInvalidValue;
    if (sw) {
        // gate/up bank [E][2][inter][k/2] (and its scales) as 5-D {k, 16 rows, gate/up,
        // 16-row block, expert}: one box {W slot, 16, 2, 4, 1} is a weight slot's eight
        // 16-row boxes in slot order (block-major, gate before up)
        auto fn = encode_fn();
        if (!fn)
            return cudaErrorInvalidValue;
        const uint64_t rb = (uint64_t)p.k / 2, rs = (uint64_t)p.k / 16, in = (uint64_t)sw->inter;
        cuuint64_t dims[5] = {rb, 16, 2, in / 16, (cuuint64_t)p.E};
        cuuint64_t strides[4] = {rb, in * rb, 16 * rb, (uint64_t)p.n * rb};
        cuuint32_t box[5] = {(cuuint32_t)(W_KS * BK / 2), 16, 2, 4, 1};
        cuuint32_t es[5] = {1, 1, 1, 1, 1};
        cuuint64_t sdims[5] = {rs, 16, 2, in / 16, (cuuint64_t)p.E};
        cuuint64_t sstrides[4] = {rs, in * rs, 16 * rs, (uint64_t)p.n * rs};
        cuuint32_t sbox[5] = {16, 16, 2, 4, 1};
        if (fn(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t *>(p.w), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            fn(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t *>(p.sc), sdims, sstrides,
               sbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w, (uint64_t)p.k / 2,
                         (uint64_t)p.E * p.n, W_KS * BK / 2, wbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
               !make_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.sc, (uint64_t)p.k / 16,
                         (uint64_t)p.E * p.n, 16, wbox, CU_TENSOR_MAP_SWIZZLE_NONE)) {
        return cudaErrorInvalidValue;
    }
    Params kp;
    kp.offsets = p.offsets;
    kp.E = p.E;
    kp.P = p.P;
    kp.n = p.n;
    kp.k = p.k;
    kp.mt = sw ? (int)(sw->inter / 64) : (p.n + BM - 1) / BM;
    kp.scale2 = p.scale2;
    kp.scale2_host = p.scale2_host;
    kp.route_flag = l.route_flag;
    kp.rowscale = l.rowscale;
    kp.out = sw ? sw->h : p.out;
    kp.err = p.err;
    kp.stall = 0;
    kp.wait_limit = take_stall_request(&kp.stall);
    kp.inter = sw ? (int)sw->inter : 0;
    kp.limit = sw ? sw->limit : 0.0f;
    // output [P, n] f32 as a tensor map with 32-row boxes of one epilogue warp's 32 columns
    // (not under SwiGLU); without one (a row stride that is not a multiple of 16 bytes)
    // every value is stored from registers
    alignas(64) CUtensorMap tmO = {};
    kp.tma_out = !sw && kp.out && p.n % 4 == 0 &&
                 (reinterpret_cast<uintptr_t>(kp.out) & 15) == 0 && p.P > 0 &&
                 p.P < ((int64_t)1 << 31) &&
                 make_map(&tmO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kp.out, (uint64_t)p.n,
                          (uint64_t)p.P, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    auto kern = sw ? tc_gemm_kernel<true> : tc_gemm_kernel<false>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[sw ? 1 : 0][dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            attr_set[sw ? 1 : 0][dev] = true;
    }
    const int64_t max_tiles = ((p.P + BN - 1) / BN + p.E) * (int64_t)kp.mt;
    const int grid = (int)(max_tiles < sms ? max_tiles : sms);
    kern<<<grid, kThreads, SMEM_BYTES, s>>>(tmB, tmW, tmS, tmO, kp);
    return cudaGetLastError();
}

// Summation depth for the tensor-core path: one f32 rounding per K=16 MMA step into the
// TMEM accumulator (k/16 steps, products exact), one for the scale2 multiply in the
// epilogue and one for the f32 rounding of ws = e4m3 * scale2 that the f64 reference
// applies per group but this path does not.
double tc_error_ops(int recipe, int64_t k)
{
    return (double)(k / 16) + (recipe == FP4_NVFP4 ? 2.0 : 0.0) + 1.0;
}

} // namespace fp4moe

// ------------------------------------------------------------------ allocation-free variant
//
// Some callers cannot call cudaMalloc: a host framework that owns every device byte and
// forbids libraries to allocate, a real-time serving loop with a no-allocation rule after
// start-up, or code whose allocator would synchronise the device at the wrong moment. For
// them the tensor-core path can run with its workspace in a fixed, file-scope device
// array instead of caller memory. The array is part of this library's image, so every
// GPU that loads the library holds it until the process exits.

namespace fp4moe {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device, looked up once per device
// (in host code the array's name is only a stand-in, never a device address).
static uint8_t *noalloc_scratch(cudaError_t *status)
{
    static std::mutex mu;
    static uint8_t *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        *status = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            *status = e;
            return nullptr;
        }
        addr[dev] = static_cast<uint8_t *>(p);
    }
    *status = cudaSuccess;
    return addr[dev];
}

void set_last_error(const char *msg);

} // namespace fp4moe

extern "C" int fp4_grouped_expert_gemm_noalloc(const float *x, int64_t num_tokens,
                                               const int32_t *row_ids, const int32_t *offsets,
                                               int num_experts, int64_t total_rows,
                                               const uint8_t *w, const uint8_t *wscale,
                                               const float *scale2, int recipe, float *out,
                                               int64_t n, int64_t k, void *stream)
{
    using namespace fp4moe;
    if ((recipe != FP4_NVFP4 && recipe != FP4_MXFP4) || num_experts < 1 ||
        num_experts > 65535 || num_tokens < 0 || total_rows < 0 || n < 0 || k < 0)
        return FP4_ERR_ARG;
    if (k == 0 || k % 128 != 0 || n == 0 || k > (1 << 20) || n > (1 << 24) ||
        total_rows > ((int64_t)1 << 31))
        return FP4_ERR_SHAPE;
    if (total_rows == 0)
        return FP4_OK;
    if (!x || !offsets || !w || !wscale || !out || (recipe == FP4_NVFP4 && !scale2))
        return FP4_ERR_ARG;
    if (!row_ids && num_tokens < total_rows)
        return FP4_ERR_SHAPE;
    auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0u; };
    if (!a16(x) || !a16(w) || !a16(wscale) || !a16(out))
        return FP4_ERR_ALIGN;
    if (!tc_supported(n, k, recipe, num_experts))
        return FP4_ERR_SHAPE;
    if (recipe == FP4_MXFP4 && !mx_supported(n, k, num_experts, w))
        return FP4_ERR_ALIGN;
    const size_t need = recipe == FP4_MXFP4 ? mx_workspace_bytes(num_tokens, total_rows, k)
                                            : tc_workspace_bytes(num_tokens, total_rows, k, recipe);
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "fp4_grouped_expert_gemm_noalloc: the call needs %zu bytes of scratch "
                 "(fp4_grouped_workspace_size), the fixed "
                 "scratch holds %zu",
                 need, kNoAllocScratchBytes);
        set_last_error(msg);
        return FP4_ERR_WORKSPACE;
    }
    cudaError_t st = cudaSuccess;
    uint8_t *scratch = noalloc_scratch(&st);
    if (!scratch) {
        char msg[256];
        snprintf(msg, sizeof(msg), "scratch address lookup failed: %s", cudaGetErrorString(st));
        set_last_error(msg);
        return FP4_ERR_LAUNCH;
    }
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
    p.err = device_error_word();
    if (!p.err)
        return FP4_ERR_LAUNCH;
    const bool mxr = recipe == FP4_MXFP4;
    cudaError_t e = mxr ? launch_mx_quantize(p, scratch, (cudaStream_t)stream)
                        : launch_tc_quantize(p, scratch, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = mxr ? launch_mx_gemm(p, scratch, (cudaStream_t)stream)
                : launch_tc_gemm(p, scratch, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
        set_last_error(msg);
        return FP4_ERR_LAUNCH;
    }
    return FP4_OK;
}
