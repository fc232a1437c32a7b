// routing.cu -- the steps around the grouped projection: the softmax top-k router, the
// CSR construction of the routed rows, and the weighted combine of their outputs back to
// tokens.
//
// CSR offsets (memra-engine 0.71.0, src/bin/kernel_check.rs, grouped MoE GEMM section):
// offsets[e+1] = offsets[e] + rows routed to expert e; within an expert the routed rows
// are in token order. The construction is deterministic (no atomics decide an order):
//   1. a bitmap per expert with one bit per token, set for every (token, slot) pair;
//   2. per expert, the running popcount of its bitmap words (one warp per expert);
//   3. offsets = the exclusive scan of the experts' row counts (one CTA);
//   4. each pair's routed row = offsets[e] + the tokens before it in e's bitmap.
// The router (memra-engine 0.125.0, src/bin/qwen4exp_gpu_gate.rs, device-router arm:
// selected ids and their order exact, weights within a few ulps) does not print its body;
// the reading taken: the topk largest logits (ties to the lower expert id), best first,
// with softmax weights over all experts or, with renormalize, over the selected ones.
// Combine (same section of kernel_check.rs: a per-routed-row factor on the output, here
// summed per token): y[t] = sum_j weight[t][j] * out[pair_rows[t][j]], fmaf in slot order.
#include "common.cuh"

#include <float.h>

namespace fp4moe {

// ------------------------------------------------------------------ router

// One warp per token; lane l holds the logits of experts l, l + 32, ... (PER_LANE of them).
template <int PER_LANE>
__global__ void __launch_bounds__(256) route_topk_kernel(const float *__restrict__ logits,
                                                         int64_t T, int E, int topk,
                                                         int renormalize, int32_t *__restrict__ ids,
                                                         float *__restrict__ weights)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
         t += warps) {
        const float *row = logits + t * E;
        float v[PER_LANE];
        float mx = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? __ldg(row + e) : -FLT_MAX;
            if (e < E)
                mx = fmaxf(mx, v[i]);
        }
        mx = warp_max(mx);
        float sum = 0.0f;  // sum over all experts of exp(l - max)
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i)
            if (lane + 32 * i < E)
                sum += expf(v[i] - mx);
        sum = warp_sum(sum);
        uint32_t taken = 0u;
        float mine = 0.0f;  // lane j keeps the logit of its selection j
        for (int j = 0; j < topk; ++j) {
            float bv = -FLT_MAX;
            int be = 0x7FFFFFFF;
#pragma unroll
            for (int i = 0; i < PER_LANE; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && (v[i] > bv || be == 0x7FFFFFFF)) {
                    bv = v[i];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
                const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
                if (oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ov > bv || (ov == bv && oe < be))) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane)
                taken |= 1u << (be >> 5);
            if (lane == j)
                mine = bv;
            if (lane == 0)
                ids[t * topk + j] = be;
        }
        const float ex = lane < topk ? expf(mine - mx) : 0.0f;
        const float denom = renormalize ? warp_sum(ex) : sum;
        if (lane < topk)
            weights[t * topk + lane] = ex / denom;
    }
}

// ------------------------------------------------------------------ CSR construction

// 1. One bit per (expert, token) pair; an id outside [0, E) or repeated within a token
//    raises FP4_DEVERR_EXPERT_ID.
__global__ void csr_bits_kernel(const int32_t *__restrict__ ids, int64_t pairs, int topk, int E,
                                int64_t words, uint32_t *__restrict__ bits, unsigned *err)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < pairs;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int e = __ldg(ids + i);
        const int64_t t = i / topk;
        if (e < 0 || e >= E) {
            raise_device_error(err, FP4_DEVERR_EXPERT_ID);
            continue;
        }
        const uint32_t bit = 1u << (t & 31);
        const uint32_t old = atomicOr(bits + (int64_t)e * words + (t >> 5), bit);
        if (old & bit)
            raise_device_error(err, FP4_DEVERR_EXPERT_ID);
    }
}

// 2. One warp per expert: prefix[e][w] = set bits of words 0 .. w-1; count[e] = all of them.
__global__ void csr_prefix_kernel(const uint32_t *__restrict__ bits, int E, int64_t words,
                                  uint32_t *__restrict__ prefix, uint32_t *__restrict__ count)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t e = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); e < E;
         e += warps) {
        uint32_t carry = 0u;
        for (int64_t w0 = 0; w0 < words; w0 += 32) {
            const int64_t w = w0 + lane;
            const uint32_t c = w < words ? __popc(bits[e * words + w]) : 0u;
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o)
                    incl += u;
            }
            if (w < words)
                prefix[e * words + w] = carry + incl - c;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0)
            count[e] = carry;
    }
}

// 3. One CTA: offsets = exclusive scan of the counts, offsets[E] = the routed rows.
__global__ void __launch_bounds__(1024) csr_offsets_kernel(const uint32_t *__restrict__ count, int E,
                                                           int32_t *__restrict__ offsets)
{
    __shared__ uint32_t warp_tot[32];
    __shared__ uint32_t base;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0)
        base = 0u;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += 1024) {
        const int e = e0 + threadIdx.x;
        const uint32_t c = e < E ? count[e] : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += u;
        }
        if (lane == 31)
            warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const uint32_t wt = warp_tot[lane];
            uint32_t wi = wt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, wi, o);
                if (lane >= o)
                    wi += u;
            }
            warp_tot[lane] = wi - wt;  // exclusive over warps
        }
        __syncthreads();
        if (e < E)
            offsets[e] = (int32_t)(base + warp_tot[warp] + incl - c);
        __syncthreads();
        if (threadIdx.x == 1023)
            base += warp_tot[31] + incl;  // the last thread's inclusive total of this chunk
        __syncthreads();
    }
    if (threadIdx.x == 0)
        offsets[E] = (int32_t)base;
}

// 4. Routed row of each pair: offsets[e] + tokens before it in expert e's bitmap.
__global__ void csr_scatter_kernel(const int32_t *__restrict__ ids, int64_t pairs, int topk, int E,
                                   int64_t words, const uint32_t *__restrict__ bits,
                                   const uint32_t *__restrict__ prefix,
                                   const int32_t *__restrict__ offsets,
                                   int32_t *__restrict__ row_ids, int32_t *__restrict__ pair_rows)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < pairs;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int e = __ldg(ids + i);
        if (e < 0 || e >= E)
            continue;
        const int64_t t = i / topk;
        const int64_t wi = (int64_t)e * words + (t >> 5);
        const uint32_t below = bits[wi] & ((1u << (t & 31)) - 1u);
        const int64_t p = (int64_t)offsets[e] + prefix[wi] + __popc(below);
        if (p < pairs) {
            row_ids[p] = (int32_t)t;
            if (pair_rows)
                pair_rows[i] = (int32_t)p;
        }
    }
}

// ------------------------------------------------------------------ combine

// y[t][c .. c+3] = sum over the token's slots j (in order) of weight * out[row][c .. c+3].
__global__ void __launch_bounds__(256) moe_combine_kernel(const float *__restrict__ out,
                                                          const int32_t *__restrict__ pair_rows,
                                                          const float *__restrict__ weights,
                                                          int64_t T, int topk, int64_t n,
                                                          int64_t P, float *__restrict__ y,
                                                          unsigned *err)
{
    const int64_t n4 = n / 4;
    const int64_t per_row = (n4 + blockDim.x - 1) / blockDim.x;  // CTAs per token row
    for (int64_t b = blockIdx.x; b < T * per_row; b += gridDim.x) {
        const int64_t t = b / per_row;
        const int64_t c4 = (b - t * per_row) * blockDim.x + threadIdx.x;
        if (c4 >= n4)
            continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < topk; ++j) {
            const int32_t r = __ldg(pair_rows + t * topk + j);
            if (r < 0 || r >= P) {
                if (c4 == 0)
                    raise_device_error(err, FP4_DEVERR_ROW_ID);
                continue;
            }
            const float wj = __ldg(weights + t * topk + j);
            const float4 o = __ldcs(reinterpret_cast<const float4 *>(out + (int64_t)r * n) + c4);
            acc.x = fmaf(wj, o.x, acc.x);
            acc.y = fmaf(wj, o.y, acc.y);
            acc.z = fmaf(wj, o.z, acc.z);
            acc.w = fmaf(wj, o.w, acc.w);
        }
        reinterpret_cast<float4 *>(y + t * n)[c4] = acc;
    }
}

// ------------------------------------------------------------------ launchers

static int sm_count()
{
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

cudaError_t launch_route_topk(const float *logits, int64_t T, int E, int topk, int renormalize,
                              int32_t *ids, float *weights, cudaStream_t s)
{
    const int64_t want = (T + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    const int blocks = (int)(want < cap ? want : cap);
    const int per = (E + 31) / 32;
    if (per <= 8)
        route_topk_kernel<8><<<blocks, 256, 0, s>>>(logits, T, E, topk, renormalize, ids, weights);
    else if (per <= 16)
        route_topk_kernel<16><<<blocks, 256, 0, s>>>(logits, T, E, topk, renormalize, ids, weights);
    else
        route_topk_kernel<32><<<blocks, 256, 0, s>>>(logits, T, E, topk, renormalize, ids, weights);
    return cudaGetLastError();
}

size_t route_csr_workspace_bytes(int64_t T, int E)
{
    const int64_t words = (T + 31) / 32;
    return ((size_t)2 * (size_t)E * (size_t)words + (size_t)E) * sizeof(uint32_t);
}

cudaError_t launch_route_csr(const int32_t *ids, int64_t T, int topk, int E, int32_t *offsets,
                             int32_t *row_ids, int32_t *pair_rows, void *workspace,
                             unsigned *err, cudaStream_t s)
{
    const int64_t words = (T + 31) / 32;
    uint32_t *bits = static_cast<uint32_t *>(workspace);
    uint32_t *prefix = bits + (int64_t)E * words;
    uint32_t *count = prefix + (int64_t)E * words;
    const int64_t pairs = T * topk;
    const int sms = sm_count();
    cudaError_t e = cudaMemsetAsync(bits, 0, (size_t)E * (size_t)words * sizeof(uint32_t), s);
    if (e != cudaSuccess)
        return e;
    const int64_t pb = (pairs + 255) / 256;
    const int pblocks = (int)(pb < (int64_t)sms * 8 ? pb : (int64_t)sms * 8);
    if (pairs > 0)
        csr_bits_kernel<<<pblocks, 256, 0, s>>>(ids, pairs, topk, E, words, bits, err);
    const int64_t eb = ((int64_t)E + 7) / 8;
    const int eblocks = (int)(eb < (int64_t)sms * 8 ? eb : (int64_t)sms * 8);
    csr_prefix_kernel<<<eblocks, 256, 0, s>>>(bits, E, words, prefix, count);
    csr_offsets_kernel<<<1, 1024, 0, s>>>(count, E, offsets);
    if (pairs > 0)
        csr_scatter_kernel<<<pblocks, 256, 0, s>>>(ids, pairs, topk, E, words, bits, prefix,
                                                   offsets, row_ids, pair_rows);
    return cudaGetLastError();
}

cudaError_t launch_moe_combine(const float *out, const int32_t *pair_rows, const float *weights,
                               int64_t T, int topk, int64_t n, int64_t P, float *y, unsigned *err,
                               cudaStream_t s)
{
    const int64_t per_row = (n / 4 + 255) / 256;
    const int64_t want = T * per_row;
    const int64_t cap = (int64_t)sm_count() * 16;
    const int blocks = (int)(want < cap ? want : cap);
    moe_combine_kernel<<<blocks, 256, 0, s>>>(out, pair_rows, weights, T, topk, n, P, y, err);
    return cudaGetLastError();
}

} // namespace fp4moe
