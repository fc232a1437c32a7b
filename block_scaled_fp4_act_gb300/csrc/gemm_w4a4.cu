// gemm_w4a4.cu -- the W4A4 NVFP4 variant: E2M1 activations with two-level scaling against
// NVFP4 weights, on the block-scaled 4-bit tensor-core MMA (tcgen05.mma
// kind::mxf4nvf4.block_scale.scale_vec::4X: one e4m3 scale per 16 k on each operand).
//
// Method (memra-engine 0.71.0, src/bin/kernel_check.rs, the NVFP4 W4A4 MMQ GEMM section):
// each activation row gets a row scale r from its amax (applied after the sum) and, per 16
// values, an e4m3 micro-scale of amax_sub / 6 taken on the row-normalised values; the
// values become E2M1 codes. With the reading stated here (the page prints no formula):
//   r = amax_row / 2688 (f32; 2688 = 6 * 448), y = x / r, s = e4m3(max|y| over 16 / 6),
//   code = E2M1 nearest to y / S (S the value of s), ties to the even code, saturating at 6,
//   sign kept; a zero row has r = 0 and zero codes and scales.
//   out[p, c] = (sum_k E2M1(a_pk) S_a(p, k/16) E2M1(w_ck) S_w(c, k/16)) * r_p * scale2_e
// Every product is exact in the MMA's own formats (E2M1 operands, ue4m3 block scales; the
// weight scales are the NVFP4 e4m3 bytes, non-negative); the sum is the tensor core's f32
// accumulation; r and scale2 are two f32 multiplies in the epilogue.
//
// Scale factors in tensor memory: one 32-bit word per row and MMA holds the four e4m3
// bytes of the MMA's 64 k (byte i for the i-th 16-group). Weight row m of MMA kk sits at
// lane m, column slot + 4 kk + m / 32; routed row n of MMA kk sits, in every 32-lane
// quarter q, at lane 32 q + n % 32, column slot + 16 + 8 kk + n / 32 (the per-quarter
// layout the MXFP4 kernel measured, with all four bytes of the word in use).
//
// Kernel structure: persistent, one CTA (16 warps) per SM, tiles (expert, 160-row block of
// its routed rows, 128-row block of its weights), the warp roles of the MXFP4 kernel:
//   warp 0   TMA producer of the packed activation codes (k-block-major boxes, 128-byte
//            swizzle) and of each stage's activation scale box [160 rows][16 bytes]
//   warp 1   MMA issuer (one elected lane issues four MMAs of K = 64 per 256-k stage)
//   warp 2   TMA producer of the weight stage (packed E2M1 box + the weight scale box)
//   warp 3   relay: waits for a stage's operands and scale factors, releases it to warp 1
//   4 - 7    epilogue: tcgen05.ld of the accumulator, x r x scale2, coalesced f32 stores
//   8 - 15   scale-factor warps (two turns of four, one per lane quarter): read the stage's
//            scale bytes from shared memory and write the words into a tensor-memory ring
// Every mbarrier wait is bounded; the abort protocol is the other tensor-core kernels'.
// Rings (measured on GB300 at the prefill shapes): the weights stream from HBM about 2 us
// away under load, so the weight ring is the deepest (7 stages, 126 KB; 4 stages were 5%
// slower); activation slots are 20 KB, the size of the largest box. The GEMM moves its
// operands as TMA boxes of 16-20 KB; on this GPU a CTA completes about one such box per
// 270 ns from L2, which with the HBM latency sets the stage rate (~0.4 us per 256 k).
#include "common.cuh"
#include "tcgen05.cuh"
#include "tma_host.h"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace fp4moe {
namespace w4a4 {

using namespace tc;

constexpr int BM = 128;
constexpr int BN = 160;
constexpr int BK = 256;              // k per stage: four MMAs of K = 64
constexpr int BKB = BK / 2;          // bytes of one row's stage (packed E2M1)
constexpr int W_STAGES = 7;          // weight stages: E2M1 box (16 KB) + scale box (2 KB)
constexpr int B_STAGES = 4;          // activation code slots (k-block-major)
constexpr int SB_STAGES = 4;         // activation scale boxes
constexpr int SF_STAGES = 4;         // scale-factor slots in tensor memory
constexpr int kMaxExperts = 1024;
constexpr int kSfTurns = 2;
constexpr int kThreads = (8 + 4 * kSfTurns) * 32;
constexpr int kWarpB = 0, kWarpMma = 1, kWarpW = 2, kWarpRelay = 3;
constexpr int A_BYTES = BM * BKB;
constexpr int SC_BYTES = BM * 16;    // 16 e4m3 bytes (256 k) per weight row
constexpr int W_BYTES = A_BYTES + SC_BYTES;
constexpr int B_BYTES = BN * BKB;      // one code slot: 32 rows x 4 k-blocks, 64 x 2, 128 or 160 x 1
constexpr int SB_BYTES = BN * 16;      // one stage's activation scales: 16 bytes per row
constexpr int OFF_W = B_STAGES * B_BYTES;
constexpr int OFF_SB = OFF_W + W_STAGES * W_BYTES;
constexpr int RING_BYTES = OFF_SB + SB_STAGES * SB_BYTES;
constexpr int NUM_BARS = 2 * (W_STAGES + B_STAGES + SB_STAGES + SF_STAGES) + 2 + 2 + 1;
// tensor memory: two f32 accumulators of BN columns, then the scale-factor ring
constexpr int kSfCol = 2 * BN;
constexpr int kSfSlotCols = 48;      // A words: 4 MMAs x 4 columns; B words: 4 x 8
static_assert(kSfCol + SF_STAGES * kSfSlotCols <= 512, "tensor memory budget");
constexpr int kNamedReady = 1;
constexpr int kNamedThreads = 64;
static_assert(kNamedReady + SF_STAGES <= 16, "named barrier ids");
constexpr int kTileInfo = SF_STAGES;
static_assert(2 * kTileInfo > SF_STAGES, "tile info ring depth");
constexpr int SMEM_BYTES =
    1024 + RING_BYTES + NUM_BARS * 8 + 16 + (kMaxExperts + 1) * 4 + kTileInfo * 4;
static_assert(B_BYTES % 1024 == 0 && W_BYTES % 1024 == 0 && OFF_W % 1024 == 0, "alignment");
static_assert(A_BYTES % 1024 == 0 && OFF_SB % 16 == 0 && SB_BYTES % 16 == 0, "alignment");
static_assert(BN * BKB <= B_BYTES && 32 * 4 * BKB <= B_BYTES && BN % 16 == 0 && BN <= 8 * 32,
              "activation box");
static_assert(BK == 4 * 64, "a stage is the four K = 64 MMAs of mma_stage_nvf4");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(kThreads <= 1024, "block size");

struct Params {
    const int32_t *offsets;
    int E;
    int64_t P;
    int n;
    int k;
    int mt;
    const float *rowscale;  // [P] f32, r of each routed row
    const float *scale2;    // [E] f32
    float *out;
    unsigned *err;
    // bounded-wait limit in clock64 cycles; stall != 0 (a test request) makes the first
    // scale-factor warp of CTA 0 withhold its first arrival, so the launch times out
    long long wait_limit;
    int stall;
};

__device__ __forceinline__ int64_t offset_at(const Params &p, int e)
{
    return p.offsets ? (int64_t)__ldg(p.offsets + e) : (e == 0 ? 0 : p.P);
}

struct Tile {
    int e;
    int m;
    int64_t row0;
    int rows;
};

__device__ __forceinline__ Tile tile_at(int t, const int *prefix, const Params &p)
{
    int lo = 0, hi = p.E;
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
    const int j = local / p.mt;
    tl.m = local - j * p.mt;
    const int64_t r0 = offset_at(p, lo), r1 = offset_at(p, lo + 1);
    tl.row0 = r0 + (int64_t)j * BN;
    const int64_t left = r1 - tl.row0;
    tl.rows = (int)(left < BN ? left : BN);
    return tl;
}

__device__ __forceinline__ int bmap_index(int rows)
{
    return rows <= 32 ? 0 : rows <= 64 ? 1 : rows <= 128 ? 2 : 3;
}
__host__ __device__ constexpr int bmap_rows(int bi) { return bi < 3 ? 32 << bi : BN; }
__host__ __device__ constexpr int bmap_kblocks(int bi) { return bi < 2 ? 4 >> bi : 1; }

struct CodeMaps {
    CUtensorMap m[4];
};

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1), f32 accumulator,
// both K-major, ue4m3 block scales (scale-type bit 23 clear), scale-factor ids 0 (the
// 4X form uses the whole word).
__device__ __forceinline__ uint32_t idesc_nvf4(int n)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// One stage from one warp: a single elect.sync, then the elected lane issues the four MMAs
// (K = 64 each: descriptors advanced by 32 bytes, scale words by their column offsets) and
// the two commits. (An elect.sync per MMA costs the issuing warp about 100 cycles per MMA;
// in one block the stage issues at the MMAs' own rate.)
__device__ __forceinline__ void mma_stage_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t sf0, uint32_t first,
                                               uint32_t bar_w, uint32_t bar_sf)
{
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
                 "setp.eq.b32 p, %5, 0;\n\t"
                 "elect.sync r|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, "
                 "%2, %3, [%4], [%6], p;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %7, "
                 "%8, %3, [%9], [%10], 1;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %11, "
                 "%12, %3, [%13], [%14], 1;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %15, "
                 "%16, %3, [%17], [%18], 1;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%19];\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%20];\n\t"
                 "}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sf0), "r"(first), "r"(sf0 + 16u),
                 "l"(a_desc + 2u), "l"(b_desc + 2u), "r"(sf0 + 4u), "r"(sf0 + 24u),
                 "l"(a_desc + 4u), "l"(b_desc + 4u), "r"(sf0 + 8u), "r"(sf0 + 32u),
                 "l"(a_desc + 6u), "l"(b_desc + 6u), "r"(sf0 + 12u), "r"(sf0 + 40u),
                 "r"(bar_w), "r"(bar_sf)
                 : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    w4a4_gemm_kernel(const __grid_constant__ CodeMaps tmB, const __grid_constant__ CUtensorMap tmSB,
                     const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmS,
                     const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + RING_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *prefix = reinterpret_cast<int *>(tmem_slot + 4);
    volatile int *tile_info = prefix + kMaxExperts + 1;

    const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const uint32_t bar0 = smem_u32(bars);
    // barrier map: weight, code, scale-box and scale-factor rings (full, empty), accumulators
    auto wfull = [&](int s) { return bar0 + 8u * s; };
    auto wempty = [&](int s) { return bar0 + 8u * (W_STAGES + s); };
    constexpr int kB = 2 * W_STAGES;
    auto bfull = [&](int s) { return bar0 + 8u * (kB + s); };
    auto bempty = [&](int s) { return bar0 + 8u * (kB + B_STAGES + s); };
    constexpr int kSB = kB + 2 * B_STAGES;
    auto sbfull = [&](int s) { return bar0 + 8u * (kSB + s); };
    auto sbempty = [&](int s) { return bar0 + 8u * (kSB + SB_STAGES + s); };
    constexpr int kSF = kSB + 2 * SB_STAGES;
    auto sffull = [&](int s) { return bar0 + 8u * (kSF + s); };
    auto sfempty = [&](int s) { return bar0 + 8u * (kSF + SF_STAGES + s); };
    constexpr int kAcc = kSF + 2 * SF_STAGES;
    auto accf = [&](int b) { return bar0 + 8u * (kAcc + b); };
    auto acce = [&](int b) { return bar0 + 8u * (kAcc + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (kAcc + 4);

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
            mbar_init(wempty(s), 1 + 4);  // the MMA commit and the stage's four SF warps
        }
        for (int s = 0; s < B_STAGES; ++s) {
            mbar_init(bfull(s), 1);
            mbar_init(bempty(s), 1);
        }
        for (int s = 0; s < SB_STAGES; ++s) {
            mbar_init(sbfull(s), 1);
            mbar_init(sbempty(s), 4);
        }
        for (int s = 0; s < SF_STAGES; ++s) {
            mbar_init(sffull(s), 4);
            mbar_init(sfempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf(b), 1);
            mbar_init(acce(b), 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        prefix[0] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpMma)
        tmem_alloc(smem_u32(tmem_slot), 512);
    __syncthreads();
    if (warp == 0) {
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
    const int nkb = p.k / BK;
    uint8_t *const ringB = smem;
    uint8_t *const ringW = smem + OFF_W;
    uint8_t *const ringSB = smem + OFF_SB;

    if (warp == kWarpB) {
        // ---------------------------------------------------------- activation producer
        // Code slots (one 3-D box of kbps k-blocks) and, per stage, the scale box of the
        // tile's rows (16 bytes each; rows past P read as zeros).
        if (lane == 0) {
            int slot = 0, sslot = 0;
            uint32_t phase = 0, sphase = 0;
            uint32_t bmask = 0, bpar = 0, smask = 0, spar = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_at(t, prefix, p);
                const int bi = bmap_index(tl.rows);
                const int kbps = bmap_kblocks(bi);
                const uint32_t box_bytes = (uint32_t)(bmap_rows(bi) * kbps * BKB);
                for (int kb = 0; kb < nkb && ok; ++kb) {
                    if (kb % kbps == 0) {
                        if (!mbar_wait(bempty(slot), phase ^ 1u, abort_flag, p.err, p.wait_limit)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bfull(slot), box_bytes);
                        tma_load_3d(smem_u32(ringB + slot * B_BYTES), &tmB.m[bi], 0, (int)tl.row0,
                                    kb, bfull(slot));
                        bmask |= 1u << slot;
                        bpar = (bpar & ~(1u << slot)) | (phase << slot);
                        if (++slot == B_STAGES) {
                            slot = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!mbar_wait(sbempty(sslot), sphase ^ 1u, abort_flag, p.err, p.wait_limit)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(sbfull(sslot), SB_BYTES);
                    tma_load_2d(smem_u32(ringSB + sslot * SB_BYTES), &tmSB, kb * 16, (int)tl.row0,
                                sbfull(sslot));
                    smask |= 1u << sslot;
                    spar = (spar & ~(1u << sslot)) | (sphase << sslot);
                    if (++sslot == SB_STAGES) {
                        sslot = 0;
                        sphase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                for (int s = 0; s < B_STAGES; ++s)
                    if (bmask & (1u << s))
                        mbar_drain(bfull(s), (bpar >> s) & 1u);
                for (int s = 0; s < SB_STAGES; ++s)
                    if (smask & (1u << s))
                        mbar_drain(sbfull(s), (spar >> s) & 1u);
            }
        }
    } else if (warp == kWarpW) {
        // ---------------------------------------------------------- weight producer
        if (lane == 0) {
            int slot = 0;
            uint32_t phase = 0, mask = 0, par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_at(t, prefix, p);
                const int yw = tl.e * p.n + tl.m * BM;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(wempty(slot), phase ^ 1u, abort_flag, p.err, p.wait_limit)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dst = ringW + slot * W_BYTES;
                    mbar_arrive_expect_tx(wfull(slot), W_BYTES);
                    tma_load_2d(smem_u32(dst), &tmA, kb * BKB, yw, wfull(slot));
                    tma_load_2d(smem_u32(dst + A_BYTES), &tmS, kb * 16, yw, wfull(slot));
                    mask |= 1u << slot;
                    par = (par & ~(1u << slot)) | (phase << slot);
                    if (++slot == W_STAGES) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                for (int s = 0; s < W_STAGES; ++s)
                    if (mask & (1u << s))
                        mbar_drain(wfull(s), (par >> s) & 1u);
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------- MMA issuer
        unsigned st = 0;  // stages issued (W slot st % W_STAGES, SF slot st % SF_STAGES)
        int bslot = 0;
        int it = 0;
        const uint64_t bdesc0 = sw128_desc(smem_u32(ringB));
        const uint64_t adesc0 = sw128_desc(smem_u32(ringW));
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            named_sync(kNamedReady + (int)(st % SF_STAGES), kNamedThreads);
            const int rows = __shfl_sync(0xFFFFFFFFu, tile_info[it % kTileInfo], 0);
            if (rows < 0)
                break;
            const int nt = max(16, (rows + 15) & ~15);
            const uint32_t idesc = idesc_nvf4(nt);
            const int buf = it & 1;
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
            const int bi = bmap_index(rows);
            const int kbmask = bmap_kblocks(bi) - 1;
            const uint32_t kb_desc = (uint32_t)(bmap_rows(bi) * BKB) >> 4;
            auto stage = [&](int kb) {
                const int j = kb & kbmask;
                const int ws = (int)(st % W_STAGES), sf = (int)(st % SF_STAGES);
                tc_fence_after();
                const uint64_t adesc = adesc0 + (uint64_t)(ws * (W_BYTES >> 4));
                const uint64_t bdesc =
                    bdesc0 + (uint64_t)(bslot * (B_BYTES >> 4) + (uint32_t)j * kb_desc);
                const uint32_t sf0 = tmem_base + (uint32_t)(kSfCol + sf * kSfSlotCols);
                mma_stage_nvf4(d_tmem, adesc, bdesc, idesc, sf0, kb == 0 ? 1u : 0u, wempty(ws),
                               sfempty(sf));
                ++st;
                if (j == kbmask || kb == nkb - 1) {
                    mma_commit_warp(bempty(bslot));
                    bslot = bslot + 1 == B_STAGES ? 0 : bslot + 1;
                }
            };
            stage(0);
            for (int kb = 1; kb < nkb; ++kb) {
                named_sync(kNamedReady + (int)(st % SF_STAGES), kNamedThreads);
                stage(kb);
            }
            mma_commit_warp(accf(buf));
        }
        mma_commit_warp(drain_bar);
        warp_mbar_drain(drain_bar, 0);
    } else if (warp == kWarpRelay) {
        // ---------------------------------------------------------- relay
        // Per stage: the code slot (at a slot's first k-block), the weight stage and the
        // scale-factor slot must be full; then the stage goes to the MMA warp. An mbarrier
        // wait costs this warp a few hundred cycles even on a completed phase, so lanes
        // 0-3 test the weight and scale-factor slots of the next four stages in one
        // instruction, and the stages found full are released without further waits.
        static_assert(SF_STAGES <= W_STAGES && SF_STAGES <= 32, "relay look-ahead");
        Ring<SF_STAGES> rf;
        Ring<W_STAGES> rw;
        Ring<B_STAGES> rb;
        int it = 0;
        int ready = 0;  // stages from rf / rw on whose weight and scale-factor slots are full
        bool aborted = false, stuck = false;
        for (int t = blockIdx.x; t < total && !aborted; t += gridDim.x, ++it) {
            const Tile tl = tile_at(t, prefix, p);
            const int buf = it & 1;
            tile_info[it % kTileInfo] = tl.rows;
            bool ok = warp_mbar_wait(acce(buf), ((it >> 1) & 1) ^ 1u, abort_flag, p.err, p.wait_limit);
            const int kbmask = bmap_kblocks(bmap_index(tl.rows)) - 1;
            for (int kb = 0; kb < nkb; ++kb) {
                const int j = kb & kbmask;
                if (ok && j == 0)
                    ok = warp_mbar_wait(bfull(rb.slot), rb.phase, abort_flag, p.err, p.wait_limit);
                if (ok && ready == 0) {
                    // stage l ahead uses slots rw.slot + l and rf.slot + l (one phase later
                    // where they wrap); their previous uses were released already, so a full
                    // phase of that parity is this stage's
                    bool full_l = false;
                    if (lane < SF_STAGES) {
                        const int fsl = rf.slot + lane, wsl = rw.slot + lane;
                        full_l = mbar_test(sffull(fsl % SF_STAGES), rf.phase ^ (fsl >= SF_STAGES ? 1u : 0u)) &&
                                 mbar_test(wfull(wsl % W_STAGES), rw.phase ^ (wsl >= W_STAGES ? 1u : 0u));
                    }
                    const unsigned full_m = __ballot_sync(0xFFFFFFFFu, full_l);
                    __syncwarp();
                    ready = __ffs(~full_m) - 1;  // consecutive full stages from rf / rw
                    if (ready == 0) {
                        ok = warp_mbar_wait(wfull(rw.slot), rw.phase, abort_flag, p.err, p.wait_limit);
                        if (ok)
                            ok = warp_mbar_wait(sffull(rf.slot), rf.phase, abort_flag, p.err, p.wait_limit);
                        ready = 1;
                    }
                }
                if (!ok) {
                    aborted = true;
                    if (!warp_mbar_drain(sfempty(rf.slot), rf.phase ^ 1u)) {
                        stuck = true;
                        break;
                    }
                }
                named_arrive(kNamedReady + rf.slot, kNamedThreads);
                rf.next();
                rw.next();
                ready = ready > 0 ? ready - 1 : 0;
                if (j == kbmask || kb == nkb - 1)
                    rb.next();
            }
            if (stuck)
                break;
            if (aborted && t + (int)gridDim.x < total) {
                tile_info[(it + 1) % kTileInfo] = -1;
                if (warp_mbar_drain(sfempty(rf.slot), rf.phase ^ 1u))
                    named_arrive(kNamedReady + rf.slot, kNamedThreads);
            }
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------------- scale-factor warps
        // Warp w serves lane quarter q = w % 4 for the stages of its turn h. Weight row
        // 32 q + lane: its 16 scale bytes of the stage are the words of the four MMAs
        // (columns 4 kk + q); routed rows 32 c + lane, c < 5: their 16 bytes likewise, in
        // columns 16 + 8 kk + c.
        const int q = warp & 3, h = (warp - 8) >> 2;
        const int r = q * 32 + lane;
        const int ntiles = (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        int g = h;  // this CTA's stage sequence
        int ws = g % W_STAGES, ss = g % SB_STAGES, fs = g % SF_STAGES;
        uint32_t wph = (uint32_t)(g / W_STAGES) & 1u, sph = (uint32_t)(g / SB_STAGES) & 1u,
                 fph = (uint32_t)(g / SF_STAGES) & 1u;
        bool ok = true;
        for (int ti = 0; ti < ntiles && ok; ++ti) {
            const Tile tl = tile_at((int)blockIdx.x + ti * (int)gridDim.x, prefix, p);
            for (int kb = g - ti * nkb; kb < nkb; kb += kSfTurns) {
                if (!mbar_wait(wfull(ws), wph, abort_flag, p.err, p.wait_limit) ||
                    !mbar_wait(sbfull(ss), sph, abort_flag, p.err, p.wait_limit)) {
                    ok = false;
                    break;
                }
                const uint4 aw =
                    *reinterpret_cast<const uint4 *>(ringW + ws * W_BYTES + A_BYTES + r * 16);
                const uint8_t *sb = ringSB + ss * SB_BYTES;
                uint32_t bw[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int n = 32 * c + lane;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (c * 32 < BN && n < tl.rows)
                        v = *reinterpret_cast<const uint4 *>(sb + n * 16);
                    bw[c] = v.x;
                    bw[8 + c] = v.y;
                    bw[16 + c] = v.z;
                    bw[24 + c] = v.w;
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(wempty(ws));
                    mbar_arrive(sbempty(ss));
                }
                if (!mbar_wait(sfempty(fs), fph ^ 1u, abort_flag, p.err, p.wait_limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col = lane_base + (uint32_t)(kSfCol + fs * kSfSlotCols);
                tmem_st1(col + (uint32_t)q, aw.x);
                tmem_st1(col + 4u + (uint32_t)q, aw.y);
                tmem_st1(col + 8u + (uint32_t)q, aw.z);
                tmem_st1(col + 12u + (uint32_t)q, aw.w);
                tmem_st32(col + 16u, bw);  // waits for all of this warp's stores
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && !(p.stall && blockIdx.x == 0 && warp == 8 && g == h))
                    mbar_arrive(sffull(fs));
                g += kSfTurns;
                ws += kSfTurns;
                if (ws >= W_STAGES) {
                    ws -= W_STAGES;
                    wph ^= 1u;
                }
                ss += kSfTurns;
                if (ss >= SB_STAGES) {
                    ss -= SB_STAGES;
                    sph ^= 1u;
                }
                fs += kSfTurns;
                if (fs >= SF_STAGES) {
                    fs -= SF_STAGES;
                    fph ^= 1u;
                }
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue (warps 4-7)
        const int q = warp & 3;
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const Tile tl = tile_at(t, prefix, p);
            const int buf = it & 1;
            if (!mbar_wait(accf(buf), (it >> 1) & 1, abort_flag, p.err, p.wait_limit))
                break;
            tc_fence_after();
            const int col = tl.m * BM + q * 32 + lane;
            const bool colok = col < p.n;
            const float s2 = __ldg(p.scale2 + tl.e);
            float *orow = p.out + tl.row0 * (int64_t)p.n + col;
            for (int c0 = 0; c0 < tl.rows; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c0), v);
                // lane j holds r of routed row c0 + j
                const float rs = c0 + lane < tl.rows ? __ldg(p.rowscale + tl.row0 + c0 + lane) : 0.0f;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const float r = __shfl_sync(0xFFFFFFFFu, rs, jj);
                    if (colok && c0 + jj < tl.rows)
                        orow[(int64_t)(c0 + jj) * p.n] = (__uint_as_float(v[jj]) * r) * s2;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce(buf));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------ activation pass

// Two f32 -> two E2M1 codes in one byte (lo in the low nibble): the hardware conversion
// rounds to the nearest E2M1 value with ties to the even code, saturates at +-6 and keeps
// the sign (negative values that round to zero give 0x8), the definition's rounding.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// The codes of fl(fl(x / r) / S) for two values (the definition's two correctly rounded
// quotients), from a = x * c with c ~ 1 / (r S): a is within 8 f32 ulps of that quotient
// (c within 3, the product 1, the two divisions 2), so when a (1 - 2^-20) and a (1 + 2^-20)
// convert to the same codes, those are the codes of the quotients; otherwise (a value
// within 2^-20 of a rounding boundary, rarely) the two divisions are done.
__device__ __forceinline__ uint32_t e2m1x2_scaled(float x0, float x1, float c, float r, float S)
{
    const float a0 = x0 * c, a1 = x1 * c;
    const uint32_t lo = e2m1x2(a0 * (1.0f - 0x1p-20f), a1 * (1.0f - 0x1p-20f));
    const uint32_t hi = e2m1x2(a0 * (1.0f + 0x1p-20f), a1 * (1.0f + 0x1p-20f));
    if (lo == hi)
        return lo;
    return e2m1x2(__fdiv_rn(__fdiv_rn(x0, r), S), __fdiv_rn(__fdiv_rn(x1, r), S));
}

constexpr int kQuantThreads = 128;

// Two-level quantisation of source row s (x[rid[s]], or x[s] without row ids), one CTA
// per row: pass 1 the row amax, pass 2 per 16-block (four consecutive threads, four
// values each): the block's max|y| = fl(max|x| / r) (division is monotone, so this is the
// largest y = fl(x / r)), the micro-scale byte e4m3(max|y| / 6) and the codes of
// fl(y / S) (e2m1x2_scaled; rows with r below 2^-100, where 1 / (r S) could overflow,
// divide every value). Writes codes[s] (k/2 bytes), scales[s] (k/16 bytes) and
// rowscale[s]. Bad row ids give a zero row (r = 0) and raise FP4_DEVERR_ROW_ID.
__global__ void __launch_bounds__(kQuantThreads) w4a4_quant_kernel(
    const float *__restrict__ x, int64_t T, const int32_t *__restrict__ rid, int64_t S, int k,
    uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, float *__restrict__ rowscale,
    unsigned *err)
{
    __shared__ float red[kQuantThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31;
    const int chunks = k >> 2;
    for (int64_t s = blockIdx.x; s < S; s += gridDim.x) {
        const int64_t t = rid ? (int64_t)__ldg(rid + s) : s;
        const bool ok = t >= 0 && t < T;
        if (!ok && tid == 0)
            raise_device_error(err, FP4_DEVERR_ROW_ID);
        const float4 *xr = reinterpret_cast<const float4 *>(x + (ok ? t : 0) * (int64_t)k);
        float amax = 0.0f;
        if (ok)
            for (int c = tid; c < chunks; c += kQuantThreads) {
                const float4 v = __ldg(xr + c);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
        amax = warp_max(amax);
        if (lane == 0)
            red[tid >> 5] = amax;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < kQuantThreads / 32; ++w)
            amax = fmaxf(amax, red[w]);
        __syncthreads();  // red is rewritten by the next row
        const float r = __fdiv_rn(amax, 2688.0f);
        if (tid == 0)
            rowscale[s] = r;
        uint16_t *crow = reinterpret_cast<uint16_t *>(codes + s * (int64_t)(k >> 1));
        uint8_t *srow = scales + s * (int64_t)(k >> 4);
        const bool fast = r >= 0x1p-100f;
        const float inv_r = fast ? __frcp_rn(r) : 0.0f;
        for (int base = 0; base < chunks; base += kQuantThreads) {
            const int c = base + tid;
            const bool act = c < chunks;  // uniform over each 4-thread block (chunks % 4 == 0)
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (act && r != 0.0f)
                v = __ldg(xr + c);
            float ax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
            ax = fmaxf(ax, __shfl_xor_sync(0xFFFFFFFFu, ax, 1));
            ax = fmaxf(ax, __shfl_xor_sync(0xFFFFFFFFu, ax, 2));
            const float m = r != 0.0f ? __fdiv_rn(ax, r) : 0.0f;
            const uint32_t sbyte = e4m3x2(__fdiv_rn(m, 6.0f), 0.0f) & 0xFFu;
            const float S = e4m3_to_f32(sbyte);
            uint32_t q = 0u;
            if (S != 0.0f) {
                if (fast) {
                    const float cs = inv_r * __frcp_rn(S);
                    q = e2m1x2_scaled(v.x, v.y, cs, r, S) | (e2m1x2_scaled(v.z, v.w, cs, r, S) << 8);
                } else {
                    q = e2m1x2(__fdiv_rn(__fdiv_rn(v.x, r), S), __fdiv_rn(__fdiv_rn(v.y, r), S)) |
                        (e2m1x2(__fdiv_rn(__fdiv_rn(v.z, r), S), __fdiv_rn(__fdiv_rn(v.w, r), S)) << 8);
                }
            }
            if (act) {
                crow[c] = (uint16_t)q;
                if ((tid & 3) == 0)
                    srow[c >> 2] = (uint8_t)sbyte;
            }
        }
    }
}

// Routed row p = token row row_ids[p] of the per-token region (codes, scales, r).
__global__ void __launch_bounds__(256) w4a4_expand_kernel(
    const uint4 *__restrict__ tok_codes, const uint4 *__restrict__ tok_scales,
    const float *__restrict__ tok_rs, const int32_t *__restrict__ row_ids, int64_t T, int64_t P,
    int k, uint4 *__restrict__ codes, uint4 *__restrict__ scales, float *__restrict__ rowscale,
    unsigned *err)
{
    const int lane = threadIdx.x & 31;
    const int cchunks = k / 32;   // 16-byte chunks of a row's k/2 code bytes
    const int schunks = k / 256;  // 16-byte chunks of a row's k/16 scale bytes
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t pr = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pr < P;
         pr += warps) {
        const int64_t t = __ldg(row_ids + pr);
        const bool ok = t >= 0 && t < T;
        if (!ok && lane == 0)
            raise_device_error(err, FP4_DEVERR_ROW_ID);
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        for (int c = lane; c < cchunks; c += 32)
            __stcs(codes + pr * cchunks + c, ok ? __ldg(tok_codes + t * cchunks + c) : zero);
        for (int c = lane; c < schunks; c += 32)
            __stcs(scales + pr * schunks + c, ok ? __ldg(tok_scales + t * schunks + c) : zero);
        if (lane == 0)
            rowscale[pr] = ok ? __ldg(tok_rs + t) : 0.0f;
    }
}

} // namespace w4a4

// ------------------------------------------------------------------ host side

static size_t w4_r1024(size_t b)
{
    return (b + 1023) & ~(size_t)1023;
}

// Workspace of this path: [codes P x k/2][scales P x k/16][r P] and, when tokens repeat,
// the same three for the T token rows; each part 1024-aligned.
size_t w4a4_workspace_bytes(int64_t num_tokens, int64_t total_rows, int64_t k)
{
    auto part = [&](int64_t rows) {
        return w4_r1024((size_t)rows * (size_t)(k / 2)) + w4_r1024((size_t)rows * (size_t)(k / 16)) +
               w4_r1024((size_t)rows * 4);
    };
    size_t b = 1024 + part(total_rows);
    if (num_tokens < total_rows)
        b += part(num_tokens);
    return b;
}

struct W4Layout {
    uint8_t *codes, *scales;
    float *rs;
    uint8_t *tok_codes, *tok_scales;
    float *tok_rs;
};

static W4Layout w4_layout(const void *ws, int64_t T, int64_t P, int64_t k)
{
    W4Layout l;
    uint8_t *b = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(ws) + 1023) & ~(uintptr_t)1023);
    l.codes = b;
    l.scales = l.codes + w4_r1024((size_t)P * (size_t)(k / 2));
    l.rs = reinterpret_cast<float *>(l.scales + w4_r1024((size_t)P * (size_t)(k / 16)));
    l.tok_codes = reinterpret_cast<uint8_t *>(l.rs) + w4_r1024((size_t)P * 4);
    l.tok_scales = l.tok_codes + w4_r1024((size_t)T * (size_t)(k / 2));
    l.tok_rs = reinterpret_cast<float *>(l.tok_scales + w4_r1024((size_t)T * (size_t)(k / 16)));
    return l;
}

// The path needs k a multiple of 256 (one stage: 128 code bytes, 16 scale bytes, both whole
// TMA rows) and at most kMaxExperts experts; its TMA bases must be 16-byte aligned.
bool w4a4_supported(int64_t n, int64_t k, int E)
{
    if (k < 256 || k % 256 != 0)
        return false;
    return E >= 1 && E <= w4a4::kMaxExperts && (int64_t)E * n < ((int64_t)1 << 31) && n >= 1;
}

static bool w4_aligned16(const void *a)
{
    return (reinterpret_cast<uintptr_t>(a) & 15u) == 0;
}

static int w4_sms()
{
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

cudaError_t launch_act_quant_w4a4(const float *x, const int32_t *rid, int64_t T, int64_t S,
                                  int64_t k, uint8_t *codes, uint8_t *scales, float *rowscale,
                                  unsigned *err, cudaStream_t s)
{
    if (S <= 0)
        return cudaSuccess;
    const int64_t cap = (int64_t)w4_sms() * 16;
    const int blocks = (int)(S < cap ? S : cap);
    w4a4::w4a4_quant_kernel<<<blocks, w4a4::kQuantThreads, 0, s>>>(x, T, rid, S, (int)k, codes,
                                                                   scales, rowscale, err);
    return cudaGetLastError();
}

cudaError_t launch_w4a4_quantize(const GroupedProblem &p, void *workspace, cudaStream_t s)
{
    const bool tok = p.row_ids != nullptr && p.T < p.P;
    const W4Layout l = w4_layout(workspace, p.T, p.P, p.k);
    cudaError_t e;
    if (tok)
        e = launch_act_quant_w4a4(p.x, nullptr, p.T, p.T, p.k, l.tok_codes, l.tok_scales,
                                  l.tok_rs, p.err, s);
    else
        e = launch_act_quant_w4a4(p.x, p.row_ids, p.T, p.P, p.k, l.codes, l.scales, l.rs, p.err, s);
    if (e != cudaSuccess || !tok)
        return e;
    const int sms = w4_sms();
    const int64_t ew = (p.P + 7) / 8;
    const int eblocks = (int)(ew < (int64_t)sms * 8 ? ew : (int64_t)sms * 8);
    w4a4::w4a4_expand_kernel<<<eblocks, 256, 0, s>>>(
        reinterpret_cast<const uint4 *>(l.tok_codes), reinterpret_cast<const uint4 *>(l.tok_scales),
        l.tok_rs, p.row_ids, p.T, p.P, p.k, reinterpret_cast<uint4 *>(l.codes),
        reinterpret_cast<uint4 *>(l.scales), l.rs, p.err);
    return cudaGetLastError();
}

cudaError_t launch_w4a4_gemm(const GroupedProblem &p, const void *workspace, cudaStream_t s)
{
    using namespace w4a4;
    if (!w4a4_supported(p.n, p.k, p.E) || !w4_aligned16(p.w) || !w4_aligned16(p.sc) || !p.scale2)
        return cudaErrorInvalidValue;
    const W4Layout l = w4_layout(workspace, p.T, p.P, p.k);
    auto fn = encode_fn();
    if (!fn)
        return cudaErrorInvalidValue;
    alignas(64) CodeMaps tmB;
    alignas(64) CUtensorMap tmSB, tmA, tmS;
    for (int i = 0; i < 4; ++i) {
        // 3-D {128 bytes, rows, k-blocks} over the [P, k/2] codes, box {128, rows_i, kblocks_i}
        cuuint64_t dims[3] = {(cuuint64_t)BKB, (cuuint64_t)p.P, (cuuint64_t)(p.k / BK)};
        cuuint64_t strides[2] = {(cuuint64_t)p.k / 2, (cuuint64_t)BKB};
        cuuint32_t box[3] = {(cuuint32_t)BKB, (cuuint32_t)bmap_rows(i), (cuuint32_t)bmap_kblocks(i)};
        cuuint32_t es[3] = {1, 1, 1};
        if (fn(&tmB.m[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, l.codes, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // activation scales [P, k/16], box {16 bytes, BN rows}; weights [E n, k/2] packed, box
    // {128 bytes, 128 rows}, 128-byte swizzle; weight scales [E n, k/16], box {16, 128}
    if (!make_map(&tmSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, l.scales, (uint64_t)p.k / 16,
                  (uint64_t)p.P, 16, BN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w, (uint64_t)p.k / 2,
                  (uint64_t)p.E * p.n, BKB, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.sc, (uint64_t)p.k / 16,
                  (uint64_t)p.E * p.n, 16, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    Params kp;
    kp.offsets = p.offsets;
    kp.E = p.E;
    kp.P = p.P;
    kp.n = p.n;
    kp.k = p.k;
    kp.mt = (p.n + BM - 1) / BM;
    kp.rowscale = l.rs;
    kp.scale2 = p.scale2;
    kp.out = p.out;
    kp.err = p.err;
    kp.stall = 0;
    kp.wait_limit = take_stall_request(&kp.stall);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(w4a4_gemm_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            attr_set[dev] = true;
    }
    const int sms = w4_sms();
    const int64_t max_tiles = ((p.P + BN - 1) / BN + p.E) * (int64_t)kp.mt;
    const int grid = (int)(max_tiles < sms ? max_tiles : sms);
    w4a4_gemm_kernel<<<grid, kThreads, SMEM_BYTES, s>>>(tmB, tmSB, tmA, tmS, kp);
    return cudaGetLastError();
}

} // namespace fp4moe
