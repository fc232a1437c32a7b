// gemm_mx.cu -- MXFP4 grouped expert GEMM on the block-scaled 8-bit tensor-core MMA
// (tcgen05.mma kind::mxf8f6f4.block_scale, one scale per 32 k).
//
// Arithmetic (memra-engine 0.98.0, src/bin/dsv4_native_gemm_gate.rs, fn f64_ref, MXFP4):
// out = sum over k of e4m3(code) * 2^(m_a) * E2M1(nibble) * 2^(e - 127). Every factor is
// carried exactly by the MMA's own operand and scale formats:
//   A (M side) = weights: E2M1 nibbles as stored, staged by TMA in the padded 4-bit
//                shared-memory form (16 values in 8 bytes, then 8 bytes the MMA skips)
//   SFA        = the weight e8m0 byte of each 32-group, used as is (ue8m0)
//   B (N side) = activations: e4m3 codes
//   SFB        = the activation's power-of-two scale per 128 as ue8m0 (its biased f32
//                exponent), the same byte for the four 32-groups of a 128-block
// so every product and scaling is exact, as on the 16-bit path, but at the 8-bit MMA rate
// (K = 32 per instruction) and with no weight conversion at all.
//
// Scale factors in tensor memory (per 128-k stage, measured on GB300): for the A side,
// weight row m reads lane m at column SFA + m / 32; for the B side, each 32-lane quarter
// of the tensor core reads its own copy, so routed row n's word sits at lane 32 q + n % 32,
// column SFB + n / 32, in every quarter q; the byte of a word is chosen per MMA by the
// instruction descriptor's scale-factor id (the k-th 32-group of the stage).
//
// Kernel structure: persistent, one CTA (16 warps) per SM, the tile schedule of the 16-bit
// path (expert, 192-row block of its routed rows, 128-row block of its weights).
//   warp 0   TMA producer of activation code slots (k-block-major boxes, 128-byte swizzle)
//            and of each stage's activation scale bytes
//   warp 1   MMA issuer (whole warp, one elected lane issues four MMAs per stage)
//   warp 2   TMA producer of the weight stage (E2M1 box + the weight scale box)
//   warp 3   relay: waits for a stage's operands and scale factors, releases it to warp 1
//   4 - 7    epilogue: tcgen05.ld of the accumulator, coalesced f32 stores
//   8 - 15   scale-factor warps (two turns of four, one per lane quarter): read the stage's
//            scale bytes from shared memory and write the words into a tensor-memory ring
// Every mbarrier wait is bounded; the abort protocol is the 16-bit kernel's.
#include "common.cuh"
#include "tcgen05.cuh"
#include "tma_host.h"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace fp4moe {
namespace mx {

using namespace tc;

constexpr int BM = 128;
constexpr int BN = 192;
constexpr int BK = 128;              // k per stage: four MMAs of K = 32
constexpr int W_STAGES = 4;          // weight stages: E2M1 box (8 KB read, 16 KB placed) + scales
// Activation code slots of 48 KB (k-block-major; one TMA copy serves 2-12 k-stages): on
// GB300 three 48 KB slots with four weight stages were 1.5% faster than four 32 KB slots
// with five; a CTA completes about one TMA copy per ~270 ns whatever its size.
constexpr int B_STAGES = 3;
constexpr int SB_STAGES = 8;         // activation scale-byte stages
constexpr int SF_STAGES = 4;         // scale-factor slots in tensor memory
constexpr int kMaxExperts = 1024;
constexpr int kSfTurns = 2;          // turns of scale-factor warps
constexpr int kThreads = (8 + 4 * kSfTurns) * 32;
constexpr int kWarpB = 0, kWarpMma = 1, kWarpW = 2, kWarpRelay = 3;
constexpr int A_BYTES = BM * BK;     // 128 rows x 128 bytes (padded 4-bit form)
constexpr int A_TX = BM * BK / 2;    // bytes the E2M1 box reads (the transaction count)
constexpr int SC_BYTES = BM * 16;    // scale box: 16 e8m0 bytes (512 k) per weight row
constexpr int W_BYTES = A_BYTES + SC_BYTES;
constexpr int B_BYTES = 32 * 12 * BK; // one code slot: 32 rows x 12 k-blocks, 64 x 6, 128 x 3, 192 x 2
constexpr int SB_BYTES = 256;        // one stage's activation scale bytes (row0 rounded down)
constexpr int OFF_W = B_STAGES * B_BYTES;
constexpr int OFF_SB = OFF_W + W_STAGES * W_BYTES;
constexpr int RING_BYTES = OFF_SB + SB_STAGES * SB_BYTES;
constexpr int NUM_BARS = 2 * (W_STAGES + B_STAGES + SB_STAGES + SF_STAGES) + 2 + 2 + 1;
// tensor memory: two f32 accumulators of BN columns, then the scale-factor ring: slot s
// holds the A words at column kSfCol + 16 s (+ quarter) and the B words at + 4 (+ n / 32)
constexpr int kSfCol = 2 * BN;
constexpr int kSfSlotCols = 16;
static_assert(kSfCol + SF_STAGES * kSfSlotCols <= 512, "tensor memory budget");
constexpr int kNamedReady = 1;
constexpr int kNamedThreads = 64;
static_assert(kNamedReady + SF_STAGES <= 16, "named barrier ids");
constexpr int kTileInfo = SF_STAGES;
static_assert(2 * kTileInfo > SF_STAGES, "tile info ring depth");
constexpr int SMEM_BYTES =
    1024 + RING_BYTES + NUM_BARS * 8 + 16 + (kMaxExperts + 1) * 4 + kTileInfo * 4;
static_assert(B_BYTES % 1024 == 0 && W_BYTES % 1024 == 0 && OFF_W % 1024 == 0, "alignment");
static_assert(BN * BK <= B_BYTES && BN % 16 == 0 && BN + 15 <= SB_BYTES, "activation box");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(kThreads <= 1024, "block size");

struct Params {
    const int32_t *offsets;
    int E;
    int64_t P;
    int n;
    int k;
    int mt;
    float *out;
    unsigned *err;
    // bounded-wait limit in clock64 cycles; stall != 0 (a test request) makes the first
    // scale-factor warp of CTA 0 withhold its first arrival, so this launch times out and
    // aborts
    long long wait_limit;
    int stall;
    // fused SwiGLU (gate/up bank: rows [0, inter) gate, [inter, 2 inter) up): out is h
    // [P, inter]; a tile covers 64 h columns (16 gate + 16 up rows per lane quarter)
    int inter;
    float limit;
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
__host__ __device__ constexpr int bmap_kblocks(int bi) { return bi == 0 ? 12 : bi == 1 ? 6 : bi == 2 ? 3 : 2; }

struct CodeMaps {
    CUtensorMap m[4];
};

// Instruction descriptor of kind::mxf8f6f4 with ue8m0 block scales: A E2M1 (5), B E4M3 (0),
// f32 accumulator, both K-major; the scale-factor ids pick the byte of the scale words.
__device__ __forceinline__ uint32_t idesc_mx(int n, uint32_t sf_id)
{
    return (sf_id << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}

// One elected lane issues D[tmem] (+)= A[smem] * B[smem]^T with block scales from tensor
// memory (sfa: A words, sfb: B words).
__device__ __forceinline__ void mma_mx_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                            uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
                 "setp.ne.b32 p, %6, 0;\n\t"
                 "elect.sync r|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, "
                 "%3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7])
                 : "memory");
}

// SWIGLU: the weight maps have 16-row boxes, eight per stage (block b: gate rows when b is
// even, up rows when odd), so lane quarter q holds 16 gate rows in lanes 0-15 and the
// matching up rows in lanes 16-31 (as in the 16-bit kernel).
template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CodeMaps tmB, const __grid_constant__ CUtensorMap tmSB,
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
    // barrier map: weight, code, scale-byte and scale-factor rings (full, empty), accumulators
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
        // Code slots (one 3-D box of kbps k-blocks) and, per stage, the 256 scale bytes of
        // the rows from row0 rounded down to 16 (the x coordinate of a TMA box must be a
        // multiple of 16 bytes).
        if (lane == 0) {
            int slot = 0, sslot = 0;
            uint32_t phase = 0, sphase = 0;
            uint32_t bmask = 0, bpar = 0, smask = 0, spar = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_at(t, prefix, p);
                const int bi = bmap_index(tl.rows);
                const int kbps = bmap_kblocks(bi);
                const uint32_t box_bytes = (uint32_t)(bmap_rows(bi) * kbps * BK);
                const int x16 = (int)(tl.row0 & ~(int64_t)15);
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
                    tma_load_2d(smem_u32(ringSB + sslot * SB_BYTES), &tmSB, x16, kb, sbfull(sslot));
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
                    mbar_arrive_expect_tx(wfull(slot), A_TX + SC_BYTES);
                    if (SWIGLU) {
#pragma unroll
                        for (int b = 0; b < 8; ++b) {
                            const int yb = tl.e * p.n + (b & 1) * p.inter + tl.m * 64 + (b >> 1) * 16;
                            tma_load_2d(smem_u32(dst + b * 16 * 128), &tmA, kb * BK, yb, wfull(slot));
                            tma_load_2d(smem_u32(dst + A_BYTES + b * 16 * 16), &tmS,
                                        ((kb * BK) / 32) & ~15, yb, wfull(slot));
                        }
                    } else {
                        tma_load_2d(smem_u32(dst), &tmA, kb * BK, yw, wfull(slot));
                        tma_load_2d(smem_u32(dst + A_BYTES), &tmS, ((kb * BK) / 32) & ~15, yw,
                                    wfull(slot));
                    }
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
            const int buf = it & 1;
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
            const int bi = bmap_index(rows);
            const int kbps = bmap_kblocks(bi);
            const uint32_t kb_desc = (uint32_t)(bmap_rows(bi) * BK) >> 4;
            auto stage = [&](int kb) {
                const int j = kb % kbps;
                const int ws = (int)(st % W_STAGES), sf = (int)(st % SF_STAGES);
                tc_fence_after();
                const uint64_t adesc = adesc0 + (uint64_t)(ws * (W_BYTES >> 4));
                const uint64_t bdesc =
                    bdesc0 + (uint64_t)(bslot * (B_BYTES >> 4) + (uint32_t)j * kb_desc);
                const uint32_t sfa = tmem_base + (uint32_t)(kSfCol + sf * kSfSlotCols);
#pragma unroll
                for (int kk = 0; kk < BK / 32; ++kk)
                    mma_mx_warp(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc_mx(nt, (uint32_t)kk),
                                sfa, sfa + 4u, (kb | kk) != 0 ? 1u : 0u);
                mma_commit_warp(wempty(ws));
                mma_commit_warp(sfempty(sf));
                ++st;
                if (j == kbps - 1 || kb == nkb - 1) {
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
        // scale-factor slot must be full; then the stage goes to the MMA warp.
        Ring<SF_STAGES> rf;
        Ring<W_STAGES> rw;
        Ring<B_STAGES> rb;
        int it = 0;
        bool aborted = false, stuck = false;
        for (int t = blockIdx.x; t < total && !aborted; t += gridDim.x, ++it) {
            const Tile tl = tile_at(t, prefix, p);
            const int buf = it & 1;
            tile_info[it % kTileInfo] = tl.rows;
            bool ok = warp_mbar_wait(acce(buf), ((it >> 1) & 1) ^ 1u, abort_flag, p.err, p.wait_limit);
            const int kbps = bmap_kblocks(bmap_index(tl.rows));
            for (int kb = 0; kb < nkb; ++kb) {
                const int j = kb % kbps;
                if (ok && j == 0)
                    ok = warp_mbar_wait(bfull(rb.slot), rb.phase, abort_flag, p.err, p.wait_limit);
                if (ok)
                    ok = warp_mbar_wait(wfull(rw.slot), rw.phase, abort_flag, p.err, p.wait_limit);
                if (ok)
                    ok = warp_mbar_wait(sffull(rf.slot), rf.phase, abort_flag, p.err, p.wait_limit);
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
                if (j == kbps - 1 || kb == nkb - 1)
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
        // Warp w serves lane quarter q = w % 4 (the lanes its tcgen05.st reaches) for the
        // stages of its turn h (h, h + kSfTurns, ...). Weight row 32 q + lane: its four e8m0
        // bytes of the stage (one word, one column); routed rows 32 c + lane, c < 8: the
        // stage's activation scale byte, repeated in the word's four bytes, in column c.
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
            const int xoff = (int)(tl.row0 & 15);
            // g is the next stage of this turn; tile ti holds stages ti * nkb .. + nkb - 1
            for (int kb = g - ti * nkb; kb < nkb; kb += kSfTurns) {
                if (!mbar_wait(wfull(ws), wph, abort_flag, p.err, p.wait_limit) ||
                    !mbar_wait(sbfull(ss), sph, abort_flag, p.err, p.wait_limit)) {
                    ok = false;
                    break;
                }
                const uint8_t *w = ringW + ws * W_BYTES + A_BYTES;
                const uint32_t aw = *reinterpret_cast<const uint32_t *>(w + r * 16 + ((kb * 4) & 15));
                const uint8_t *sb = ringSB + ss * SB_BYTES + xoff;
                uint32_t bw[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int n = 32 * c + lane;
                    const uint32_t byte = n < tl.rows ? sb[n] : 127u;
                    bw[c] = byte * 0x01010101u;
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
                tmem_st1(col + (uint32_t)q, aw);
                tmem_st8(col + 4u, bw);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && !(p.stall && blockIdx.x == 0 && warp == 8 && g == h))
                    mbar_arrive(sffull(fs));
                // next stage of this turn: kSfTurns stages later
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
            // SWIGLU: lanes 0-15 own h column col, lanes 16-31 hold the matching up rows
            const int col = SWIGLU ? tl.m * 64 + q * 16 + (lane & 15) : tl.m * BM + q * 32 + lane;
            const int ldo = SWIGLU ? p.inter : p.n;
            const bool colok = SWIGLU ? (lane < 16 && col < p.inter) : col < p.n;
            float *orow = p.out + tl.row0 * (int64_t)ldo + col;
            for (int c0 = 0; c0 < tl.rows; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c0), v);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const float val = __uint_as_float(v[jj]);
                    if (SWIGLU) {
                        const float up = __shfl_xor_sync(0xFFFFFFFFu, val, 16);
                        if (colok && c0 + jj < tl.rows)
                            orow[(int64_t)(c0 + jj) * ldo] = swiglu_one(val, up, p.limit);
                    } else if (colok && c0 + jj < tl.rows) {
                        orow[(int64_t)(c0 + jj) * ldo] = val;
                    }
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

// act_quant of source row s (x[rid[s]], or x[s] without row ids) per 128-group (fn
// quant_rows of dsv4_native_gemm_gate.rs): e4m3 codes into codes[s], the group scale's
// biased f32 exponent (its ue8m0 form) into sexp[g * sp + s]. One warp per group; bad row
// ids give zero codes with a unit scale and raise FP4_DEVERR_ROW_ID.
__global__ void __launch_bounds__(256) quant_mx_kernel(const float *__restrict__ x, int64_t T,
                                                       const int32_t *__restrict__ rid, int64_t S,
                                                       int k, uint8_t *__restrict__ codes,
                                                       uint8_t *__restrict__ sexp, int64_t sp,
                                                       unsigned *err)
{
    const int lane = threadIdx.x & 31;
    const int kq = k >> 7;
    const int64_t groups = S * kq;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t gi = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); gi < groups;
         gi += warps) {
        const int64_t s = gi / kq;
        const int g = (int)(gi - s * kq);
        const int64_t t = rid ? (int64_t)__ldg(rid + s) : s;
        uint32_t qv = 0u, e = 127u;
        if (t >= 0 && t < T) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(x + t * k + g * 128) + lane);
            float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
            amax = warp_max(amax);
            const float sc = group_scale(amax);
            const float inv = pow2_reciprocal(sc);
            qv = e4m3x4(scaled_clamped(v.x, inv), scaled_clamped(v.y, inv), scaled_clamped(v.z, inv),
                        scaled_clamped(v.w, inv));
            e = __float_as_uint(sc) >> 23;
        } else if (lane == 0 && g == 0) {
            raise_device_error(err, FP4_DEVERR_ROW_ID);
        }
        reinterpret_cast<uint32_t *>(codes + s * k + g * 128)[lane] = qv;
        if (lane == 0)
            sexp[(int64_t)g * sp + s] = (uint8_t)e;
    }
}

// Routed row p = token row row_ids[p] of the per-token region (codes and scale bytes).
__global__ void __launch_bounds__(256) expand_mx_kernel(const uint4 *__restrict__ tok_codes,
                                                        const uint8_t *__restrict__ tok_sexp,
                                                        int64_t tsp, const int32_t *__restrict__ row_ids,
                                                        int64_t T, int64_t P, int k,
                                                        uint4 *__restrict__ codes,
                                                        uint8_t *__restrict__ sexp, int64_t sp,
                                                        unsigned *err)
{
    const int lane = threadIdx.x & 31;
    const int chunks = k / 16;
    const int kq = k >> 7;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t pr = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pr < P;
         pr += warps) {
        const int64_t t = __ldg(row_ids + pr);
        const bool ok = t >= 0 && t < T;
        if (!ok && lane == 0)
            raise_device_error(err, FP4_DEVERR_ROW_ID);
        const uint4 *src = tok_codes + (ok ? t : 0) * chunks;
        uint4 *dst = codes + pr * chunks;
        for (int c = lane; c < chunks; c += 32)
            __stcs(dst + c, ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u));
        for (int g = lane; g < kq; g += 32)
            sexp[(int64_t)g * sp + pr] = ok ? __ldg(tok_sexp + (int64_t)g * tsp + t) : (uint8_t)127;
    }
}

} // namespace mx

// ------------------------------------------------------------------ host side

static size_t r1024(size_t b)
{
    return (b + 1023) & ~(size_t)1023;
}

static int64_t pad16(int64_t v)
{
    return (v + 15) & ~(int64_t)15;
}

// Workspace of this path: [codes P x k][scale bytes (k/128) x pad16(P)] and, when tokens
// repeat, [codes T x k][scale bytes (k/128) x pad16(T)], each part 1024-aligned.
size_t mx_workspace_bytes(int64_t num_tokens, int64_t total_rows, int64_t k)
{
    size_t b = 1024 + r1024((size_t)total_rows * k) + r1024((size_t)(k / 128) * pad16(total_rows));
    if (num_tokens < total_rows)
        b += r1024((size_t)num_tokens * k) + r1024((size_t)(k / 128) * pad16(num_tokens));
    return b;
}

struct MxLayout {
    uint8_t *codes, *sexp, *tok_codes, *tok_sexp;
};

static MxLayout mx_layout(const void *ws, int64_t T, int64_t P, int64_t k)
{
    MxLayout l;
    l.codes = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(ws) + 1023) & ~(uintptr_t)1023);
    l.sexp = l.codes + r1024((size_t)P * k);
    l.tok_codes = l.sexp + r1024((size_t)(k / 128) * pad16(P));
    l.tok_sexp = l.tok_codes + r1024((size_t)T * k);
    return l;
}

// The path needs k a multiple of 512 (whole TMA units of the scale tensor), E2M1 rows whose
// byte stride is a multiple of 32 and a 32-byte aligned weight base (the packed 4-bit TMA
// form), and at most kMaxExperts experts.
bool mx_supported(int64_t n, int64_t k, int E, const void *w)
{
    if (k % 512 != 0 || (reinterpret_cast<uintptr_t>(w) & 31u) != 0)
        return false;
    return E >= 1 && E <= mx::kMaxExperts && (int64_t)E * n < ((int64_t)1 << 31) && n >= 1;
}

static int mx_sms()
{
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

cudaError_t launch_mx_quantize(const GroupedProblem &p, void *workspace, cudaStream_t s)
{
    using namespace mx;
    const bool tok = p.row_ids != nullptr && p.T < p.P;
    const MxLayout l = mx_layout(workspace, p.T, p.P, p.k);
    const int64_t S = tok ? p.T : p.P;
    const int sms = mx_sms();
    const int64_t groups = S * (p.k / 128);
    const int64_t want = (groups + 7) / 8;
    const int blocks = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    if (groups > 0)
        quant_mx_kernel<<<blocks, 256, 0, s>>>(p.x, p.T, tok ? nullptr : p.row_ids, S, p.k,
                                                tok ? l.tok_codes : l.codes,
                                                tok ? l.tok_sexp : l.sexp,
                                                tok ? pad16(p.T) : pad16(p.P), p.err);
    if (tok) {
        const int64_t ew = (p.P + 7) / 8;
        const int eblocks = (int)(ew < (int64_t)sms * 8 ? ew : (int64_t)sms * 8);
        expand_mx_kernel<<<eblocks, 256, 0, s>>>(reinterpret_cast<const uint4 *>(l.tok_codes),
                                                 l.tok_sexp, pad16(p.T), p.row_ids, p.T, p.P, p.k,
                                                 reinterpret_cast<uint4 *>(l.codes), l.sexp,
                                                 pad16(p.P), p.err);
    }
    return cudaGetLastError();
}

cudaError_t launch_mx_gemm(const GroupedProblem &p, const void *workspace, cudaStream_t s,
                           const SwigluOut *sw)
{
    using namespace mx;
    if (!mx_supported(p.n, p.k, p.E, p.w))
        return cudaErrorInvalidValue;
    if (sw && (sw->inter % 64 != 0 || 2 * sw->inter != p.n))
        return cudaErrorInvalidValue;
    const uint32_t wbox = sw ? 16 : BM;  // rows per weight box
    const MxLayout l = mx_layout(workspace, p.T, p.P, p.k);
    auto fn = encode_fn();
    if (!fn)
        return cudaErrorInvalidValue;
    alignas(64) CodeMaps tmB;
    alignas(64) CUtensorMap tmSB, tmA, tmS;
    for (int i = 0; i < 4; ++i) {
        // 3-D {128 k, rows, k-blocks} over the [P, k] codes, box {128, rows_i, kblocks_i}
        cuuint64_t dims[3] = {(cuuint64_t)BK, (cuuint64_t)p.P, (cuuint64_t)(p.k / BK)};
        cuuint64_t strides[2] = {(cuuint64_t)p.k, (cuuint64_t)BK};
        cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)bmap_rows(i), (cuuint32_t)bmap_kblocks(i)};
        cuuint32_t es[3] = {1, 1, 1};
        if (fn(&tmB.m[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, l.codes, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // 2-D {pad16(P) rows, k/128} scale bytes, box {256, 1}
        cuuint64_t dims[2] = {(cuuint64_t)pad16(p.P), (cuuint64_t)(p.k / BK)};
        cuuint64_t strides[1] = {(cuuint64_t)pad16(p.P)};
        cuuint32_t box[2] = {(cuuint32_t)SB_BYTES, 1};
        cuuint32_t es[2] = {1, 1};
        if (fn(&tmSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, l.sexp, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // 2-D {k E2M1 values, E n rows}, box {128 values, 128 rows}, padded 4-bit form
        cuuint64_t dims[2] = {(cuuint64_t)p.k, (cuuint64_t)p.E * p.n};
        cuuint64_t strides[1] = {(cuuint64_t)p.k / 2};
        cuuint32_t box[2] = {(cuuint32_t)BK, wbox};
        cuuint32_t es[2] = {1, 1};
        if (fn(&tmA, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t *>(p.w), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (!make_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.sc, (uint64_t)p.k / 32,
                  (uint64_t)p.E * p.n, 16, wbox, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    Params kp;
    kp.offsets = p.offsets;
    kp.E = p.E;
    kp.P = p.P;
    kp.n = p.n;
    kp.k = p.k;
    kp.mt = sw ? (int)(sw->inter / 64) : (p.n + BM - 1) / BM;
    kp.out = sw ? sw->h : p.out;
    kp.err = p.err;
    kp.stall = 0;
    kp.wait_limit = take_stall_request(&kp.stall);
    kp.inter = sw ? (int)sw->inter : 0;
    kp.limit = sw ? sw->limit : 0.0f;
    auto kern = sw ? mx_gemm_kernel<true> : mx_gemm_kernel<false>;
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
    const int sms = mx_sms();
    const int64_t max_tiles = ((p.P + BN - 1) / BN + p.E) * (int64_t)kp.mt;
    const int grid = (int)(max_tiles < sms ? max_tiles : sms);
    kern<<<grid, kThreads, SMEM_BYTES, s>>>(tmB, tmSB, tmA, tmS, kp);
    return cudaGetLastError();
}

} // namespace fp4moe
