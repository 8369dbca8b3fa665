// moe.cu -- routing, expert-grouped row layout, gather and combine of the
// Mixture-of-Experts FFN.  The expert FFNs themselves run in the engine.
//
// "Fine-Grained Compute-Communication Overlap for MoE" (review of arXiv
// 2607.19539): section 2.1 (router distribution over E experts, top-k, gate-
// weighted sum), section 2.2 steps 1, 3, 5 (routing, expert computation,
// weighted reduction), section 4.2 (rows grouped contiguously, each group
// zero-padded up to a whole tile so that every tile belongs to one group).
// On one GPU the groups are the experts, in ascending expert order, tokens
// ascending inside an expert.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace tffn {
namespace moe {

// ------------------------------------------------------------------ routing
// One thread per token: slot s takes the largest logit not yet taken, the
// lower expert index winning ties; gate weights are the softmax over the k
// kept logits.
__global__ void route_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                             int32_t* __restrict__ topk_idx, float* __restrict__ topk_w)
{
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= T)
        return;
    const float* l = logits + t * E;
    uint64_t taken = 0;
    float lmax = 0.0f;
    for (int s = 0; s < k; ++s) {
        int best = -1;
        float bv = 0.0f;
        for (int e = 0; e < E; ++e) {
            if ((taken >> e) & 1ull)
                continue;
            const float v = l[e];
            if (best < 0 || v > bv) {
                best = e;
                bv = v;
            }
        }
        taken |= 1ull << best;
        topk_idx[t * k + s] = best;
        topk_w[t * k + s] = bv;
        if (s == 0)
            lmax = bv;
    }
    float sum = 0.0f;
    for (int s = 0; s < k; ++s)
        sum += expf(topk_w[t * k + s] - lmax);
    const float inv = 1.0f / sum;
    for (int s = 0; s < k; ++s)
        topk_w[t * k + s] = expf(topk_w[t * k + s] - lmax) * inv;
}

// --------------------------------------------------------------------- plan
constexpr int PLAN_THREADS = 1024;

// Exclusive scan of one value per thread across the block; returns the
// thread's exclusive prefix and leaves the block total in *total.
__device__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_sums, int32_t* total)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o)
                s += y;
        }
        warp_sums[lane] = s;   // inclusive over warps
    }
    __syncthreads();
    const int32_t before = (warp > 0 ? warp_sums[warp - 1] : 0) + (x - v);
    *total = warp_sums[31];
    __syncthreads();
    return before;
}

// Single CTA.  Entries i = t*k + s are split into contiguous chunks, one per
// thread, so a per-expert exclusive scan over threads keeps token order.
// The experts' padded segments are laid out in expert index order, or, with
// size_desc, largest row count first (ties: lower index first), the schedule
// order of "Fine-Grained Compute-Communication Overlap for MoE", section 4.4,
// rule (ii).  The public outputs (perm, offsets) keep expert index order
// either way: they describe the grouping, not the internal layout.
__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(
    const int32_t* __restrict__ topk_idx, int64_t T, int E, int k, int bm, int size_desc,
    int32_t* __restrict__ pos, int32_t* __restrict__ row_src, int32_t* __restrict__ band_expert,
    int32_t* __restrict__ nbands, int32_t* __restrict__ perm_out, int32_t* __restrict__ offs_out)
{
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t s_total[64];
    __shared__ int32_t s_pad[64];       // first grouped row of expert e's segment
    __shared__ int32_t s_pad_end[64];   // one past its last (padding included)
    __shared__ int32_t s_off[65];
    const int64_t R = T * k;
    const int64_t chunk = (R + PLAN_THREADS - 1) / PLAN_THREADS;
    const int64_t i0 = static_cast<int64_t>(threadIdx.x) * chunk;
    const int64_t i1 = i0 + chunk < R ? i0 + chunk : R;

    int32_t cnt[64];
    for (int e = 0; e < E; ++e)
        cnt[e] = 0;
    for (int64_t i = i0; i < i1; ++i)
        ++cnt[topk_idx[i]];
    int32_t start[64];
    for (int e = 0; e < E; ++e) {
        int32_t tot;
        start[e] = block_exclusive_scan(cnt[e], warp_sums, &tot);
        if (threadIdx.x == 0)
            s_total[e] = tot;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t order[64];
        for (int e = 0; e < E; ++e) {
            // stable insertion: an expert goes after every earlier one that
            // is at least as large
            int j = e;
            if (size_desc)
                while (j > 0 && s_total[order[j - 1]] < s_total[e]) {
                    order[j] = order[j - 1];
                    --j;
                }
            order[j] = e;
        }
        int32_t p = 0;
        for (int j = 0; j < E; ++j) {
            const int e = order[j];
            s_pad[e] = p;
            p += (s_total[e] + bm - 1) / bm * bm;
            s_pad_end[e] = p;
        }
        int32_t o = 0;
        for (int e = 0; e < E; ++e) {
            s_off[e] = o;
            o += s_total[e];
        }
        s_off[E] = o;
        *nbands = p / bm;
    }
    __syncthreads();
    // Scatter: grouped row of each (token, slot) entry, and its source token.
    for (int64_t i = i0; i < i1; ++i) {
        const int e = topk_idx[i];
        const int32_t within = start[e]++;
        const int32_t r = s_pad[e] + within;
        pos[i] = r;
        row_src[r] = static_cast<int32_t>(i / k);
        if (perm_out)
            perm_out[s_off[e] + within] = static_cast<int32_t>(i);
    }
    // Padding rows read no token; bands map to their expert.
    for (int e = 0; e < E; ++e) {
        for (int32_t r = s_pad[e] + s_total[e] + threadIdx.x; r < s_pad_end[e]; r += blockDim.x)
            row_src[r] = -1;
        for (int32_t b = s_pad[e] / bm + threadIdx.x; b < s_pad_end[e] / bm; b += blockDim.x)
            band_expert[b] = e;
    }
    if (offs_out)
        for (int e = threadIdx.x; e <= E; e += blockDim.x)
            offs_out[e] = s_off[e];
}

// ------------------------------------------------------------------- gather
// One warp per grouped row: X_perm[r] = X[row_src[r]] (zeros for padding).
__global__ void gather_kernel(const __nv_bfloat16* __restrict__ X, const int32_t* __restrict__ row_src,
                              const int32_t* __restrict__ nbands, int bm, int64_t N,
                              __nv_bfloat16* __restrict__ Xp)
{
    const int64_t rows = static_cast<int64_t>(*nbands) * bm;
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t nvec = N / 8;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        const int32_t t = row_src[r];
        uint4* dst = reinterpret_cast<uint4*>(Xp + r * N);
        if (t < 0) {
            for (int64_t c = lane; c < nvec; c += 32)
                dst[c] = make_uint4(0u, 0u, 0u, 0u);
        } else {
            const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(t) * N);
            for (int64_t c = lane; c < nvec; c += 32)
                dst[c] = __ldg(src + c);
        }
    }
}

// ------------------------------------------------------------------ combine
// One warp per token: Y[t] = bf16(sum_s w[t,s] * Yp[pos[t,s]]), slots in order.
__global__ void combine_kernel(const float* __restrict__ Yp, const int32_t* __restrict__ pos,
                               const float* __restrict__ topk_w, int64_t T, int k, int64_t P,
                               __nv_bfloat16* __restrict__ Y)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t nvec = P / 4;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
         t += warps) {
        for (int64_t c = lane; c < nvec; c += 32) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s = 0; s < k; ++s) {
                const float g = topk_w[t * k + s];
                const float4 v = __ldg(reinterpret_cast<const float4*>(Yp + static_cast<int64_t>(pos[t * k + s]) * P) + c);
                acc.x = fmaf(g, v.x, acc.x);
                acc.y = fmaf(g, v.y, acc.y);
                acc.z = fmaf(g, v.z, acc.z);
                acc.w = fmaf(g, v.w, acc.w);
            }
            uint2 out = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
            reinterpret_cast<uint2*>(Y + t * P)[c] = out;
        }
    }
}

}  // namespace moe

int launch_moe_route(const float* logits, int64_t T, int E, int k, int32_t* idx, float* w,
                     cudaStream_t s)
{
    const int threads = 256;
    const int64_t blocks = (T + threads - 1) / threads;
    moe::route_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(logits, T, E, k, idx, w);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_moe_plan(const int32_t* idx, int64_t T, int E, int k, int bm, int size_desc, int32_t* pos,
                    int32_t* row_src, int32_t* band_expert, int32_t* nbands, int32_t* perm_out,
                    int32_t* offs_out, cudaStream_t s)
{
    moe::plan_kernel<<<1, moe::PLAN_THREADS, 0, s>>>(idx, T, E, k, bm, size_desc, pos, row_src, band_expert, nbands,
                                                     perm_out, offs_out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_moe_gather(const void* X, const int32_t* row_src, const int32_t* nbands, int bm, int64_t N,
                      void* Xp, int grid, cudaStream_t s)
{
    moe::gather_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(X), row_src, nbands, bm, N,
                                            static_cast<__nv_bfloat16*>(Xp));
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_moe_combine(const float* Yp, const int32_t* pos, const float* w, int64_t T, int k, int64_t P,
                       void* Y, int grid, cudaStream_t s)
{
    moe::combine_kernel<<<grid, 256, 0, s>>>(Yp, pos, w, T, k, P, static_cast<__nv_bfloat16*>(Y));
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tffn
