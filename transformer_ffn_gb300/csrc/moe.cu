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
// Tokens are taken in blocks of ROUTE_BLOCK; the block's entries (t, s) are
// ranked and copied by the same block of scatter_gather_kernel.
constexpr int ROUTE_BLOCK = 128;

// One thread per token: slot s takes the largest logit not yet taken, the
// lower expert index winning ties; gate weights are the softmax over the k
// kept logits.  Each block also counts its entries per expert (blk_hist).
__global__ void __launch_bounds__(ROUTE_BLOCK) route_kernel(const float* __restrict__ logits, int64_t T, int E,
                                                            int k, int32_t* __restrict__ topk_idx,
                                                            float* __restrict__ topk_w,
                                                            int32_t* __restrict__ blk_hist)
{
    __shared__ int32_t hist[64];
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        hist[e] = 0;
    __syncthreads();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t < T) {
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
            atomicAdd(&hist[best], 1);
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
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        blk_hist[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// --------------------------------------------------------------------- plan
// One CTA, one warp per expert (up to 32; a warp takes experts w, w + 32).
// From the per-block counts: each expert's padded segment
// (laid out in expert index order, or, with size_desc, largest row count
// first -- ties to the lower index -- the schedule order of "Fine-Grained
// Compute-Communication Overlap for MoE", section 4.4, rule (ii)), the band
// table, and for every token block the first grouped row of its entries of
// each expert (blk_pad) and their first position in the unpadded, expert-index
// order (blk_off, for the public permutation).  pad[2e], pad[2e+1]: first
// padding row of expert e and how many follow.
__global__ void plan_kernel(const int32_t* __restrict__ blk_hist, int nblk, int E, int bm, int size_desc,
                            int32_t* __restrict__ blk_pad, int32_t* __restrict__ blk_off,
                            int32_t* __restrict__ band_expert, int32_t* __restrict__ nbands,
                            int32_t* __restrict__ pad, int32_t* __restrict__ offs_out)
{
    __shared__ int32_t tot[64], s_pad[64], s_end[64], s_off[65];
    __shared__ int32_t s_nbands;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    // Each warp sums the token blocks' counts of its experts, 32 blocks at a time.
    for (int e = warp; e < E; e += nwarps) {
        int32_t c = 0;
        for (int b0 = 0; b0 < nblk; b0 += 32) {
            const int b = b0 + lane;
            int32_t v = b < nblk ? blk_hist[static_cast<int64_t>(b) * E + e] : 0;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1)
                v += __shfl_xor_sync(0xffffffffu, v, d);
            c += v;
        }
        if (lane == 0)
            tot[e] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t order[64];
        for (int x = 0; x < E; ++x) {
            // stable insertion: an expert goes after every earlier one that
            // is at least as large
            int j = x;
            if (size_desc)
                while (j > 0 && tot[order[j - 1]] < tot[x]) {
                    order[j] = order[j - 1];
                    --j;
                }
            order[j] = x;
        }
        int32_t p = 0;
        for (int j = 0; j < E; ++j) {
            const int x = order[j];
            s_pad[x] = p;
            p += (tot[x] + bm - 1) / bm * bm;
            s_end[x] = p;
        }
        int32_t o = 0;
        for (int x = 0; x < E; ++x) {
            s_off[x] = o;
            o += tot[x];
        }
        s_off[E] = o;
        s_nbands = p / bm;
        *nbands = p / bm;
    }
    __syncthreads();
    // Each block's first row in the padded and in the unpadded layout, per
    // expert: an exclusive prefix sum over the blocks in token order.
    for (int e = warp; e < E; e += nwarps) {
        int32_t rp = s_pad[e], ro = s_off[e];
        for (int b0 = 0; b0 < nblk; b0 += 32) {
            const int b = b0 + lane;
            const int64_t at = static_cast<int64_t>(b) * E + e;
            const int32_t v = b < nblk ? blk_hist[at] : 0;
            int32_t incl = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t u = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d)
                    incl += u;
            }
            if (b < nblk) {
                blk_pad[at] = rp + incl - v;
                blk_off[at] = ro + incl - v;
            }
            const int32_t chunk = __shfl_sync(0xffffffffu, incl, 31);
            rp += chunk;
            ro += chunk;
        }
        if (lane == 0) {
            pad[2 * e] = s_pad[e] + tot[e];
            pad[2 * e + 1] = s_end[e] - (s_pad[e] + tot[e]);
        }
    }
    for (int b = threadIdx.x; b < s_nbands; b += blockDim.x) {
        int x = 0;
        while (x < E - 1 && !(b * bm >= s_pad[x] && b * bm < s_end[x]))
            ++x;
        band_expert[b] = x;
    }
    if (offs_out)
        for (int x = threadIdx.x; x <= E; x += blockDim.x)
            offs_out[x] = s_off[x];
}

// ------------------------------------------------------------------ scatter
// One block per token block.  Warp 0 ranks the block's entries i = t*k + s in
// order (a warp-wide match of the expert ids of 32 consecutive entries gives
// each its rank among the equal ones; a running count per expert carries the
// rank across groups), which keeps (expert, token) order stably.
__global__ void __launch_bounds__(32) scatter_kernel(const int32_t* __restrict__ topk_idx, int64_t T, int E, int k,
                                                     const int32_t* __restrict__ blk_pad,
                                                     const int32_t* __restrict__ blk_off, int32_t* __restrict__ pos,
                                                     int32_t* __restrict__ perm_out, int32_t* __restrict__ row_entry)
{
    __shared__ int32_t cnt[64];
    const int lane = threadIdx.x;
    const int64_t b = blockIdx.x;
    const int64_t i0 = b * ROUTE_BLOCK * k;
    const int64_t R = T * k;
    const int n_ent = static_cast<int>(i0 + ROUTE_BLOCK * k <= R ? ROUTE_BLOCK * k : R - i0);
    cnt[lane] = 0;
    cnt[lane + 32] = 0;
    __syncwarp();
    for (int c = 0; c < n_ent; c += 32) {
        const int j = c + lane;
        const bool valid = j < n_ent;
        const int e = valid ? topk_idx[i0 + j] : -1;
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & ((1u << lane) - 1u));
        const int32_t base = valid ? cnt[e] : 0;
        if (valid) {
            const int32_t r = blk_pad[b * E + e] + base + rank;
            pos[i0 + j] = r;
            if (row_entry)
                row_entry[r] = static_cast<int32_t>(i0 + j);
            if (perm_out)
                perm_out[blk_off[b * E + e] + base + rank] = static_cast<int32_t>(i0 + j);
        }
        __syncwarp();
        if (valid && lane == __ffs(same) - 1)
            cnt[e] = base + __popc(same);
        __syncwarp();
    }
}

// ------------------------------------------------------------------- gather
// One warp per entry: X_perm[pos[i]] = X[i / k]; then the experts' padding
// rows (pad[2e] first row, pad[2e+1] count), numbered across experts, are
// zeroed, one per warp, and marked -1 in row_entry (when given).
__global__ void gather_kernel(const __nv_bfloat16* __restrict__ X, const int32_t* __restrict__ pos, int64_t R, int k,
                              const int32_t* __restrict__ pad, int E, int64_t N, __nv_bfloat16* __restrict__ Xp,
                              int32_t* __restrict__ row_entry)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t w0 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nvec = N / 8;   // 16-byte vectors per row
    for (int64_t i = w0; i < R; i += warps) {
        const uint4* src = reinterpret_cast<const uint4*>(X + (i / k) * N);
        uint4* dst = reinterpret_cast<uint4*>(Xp + static_cast<int64_t>(pos[i]) * N);
        for (int64_t c = lane; c < nvec; c += 32)
            dst[c] = __ldg(src + c);
    }
    int64_t total = 0;
    for (int e = 0; e < E; ++e)
        total += pad[2 * e + 1];
    for (int64_t q = w0; q < total; q += warps) {
        int e = 0;
        int64_t rest = q;
        while (rest >= pad[2 * e + 1]) {
            rest -= pad[2 * e + 1];
            ++e;
        }
        uint4* dst = reinterpret_cast<uint4*>(Xp + (pad[2 * e] + rest) * N);
        for (int64_t c = lane; c < nvec; c += 32)
            dst[c] = make_uint4(0u, 0u, 0u, 0u);
        if (row_entry && lane == 0)
            row_entry[pad[2 * e] + rest] = -1;
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

int moe_route_blocks(int64_t T)
{
    return static_cast<int>((T + moe::ROUTE_BLOCK - 1) / moe::ROUTE_BLOCK);
}

int launch_moe_route(const float* logits, int64_t T, int E, int k, int32_t* idx, float* w, int32_t* blk_hist,
                     cudaStream_t s)
{
    moe::route_kernel<<<moe_route_blocks(T), moe::ROUTE_BLOCK, 0, s>>>(logits, T, E, k, idx, w, blk_hist);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_moe_plan(const int32_t* blk_hist, int64_t T, int E, int bm, int size_desc, int32_t* blk_pad,
                    int32_t* blk_off, int32_t* band_expert, int32_t* nbands, int32_t* pad, int32_t* offs_out,
                    cudaStream_t s)
{
    const int warps = E < 32 ? E : 32;   // one warp per expert, up to 32
    moe::plan_kernel<<<1, 32 * warps, 0, s>>>(blk_hist, moe_route_blocks(T), E, bm, size_desc, blk_pad, blk_off,
                                              band_expert, nbands, pad, offs_out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_moe_scatter(const int32_t* idx, int64_t T, int E, int k, const int32_t* blk_pad, const int32_t* blk_off,
                       int32_t* pos, int32_t* perm_out, int32_t* row_entry, cudaStream_t s)
{
    moe::scatter_kernel<<<moe_route_blocks(T), 32, 0, s>>>(idx, T, E, k, blk_pad, blk_off, pos, perm_out, row_entry);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_moe_gather(const void* X, const int32_t* pos, int64_t T, int k, const int32_t* pad, int E, int64_t N,
                      void* Xp, int32_t* row_entry, int grid, cudaStream_t s)
{
    moe::gather_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(X), pos, T * k, k, pad, E, N,
                                            static_cast<__nv_bfloat16*>(Xp), row_entry);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_moe_combine(const float* Yp, const int32_t* pos, const float* w, int64_t T, int k, int64_t P,
                       void* Y, int grid, cudaStream_t s)
{
    moe::combine_kernel<<<grid, 256, 0, s>>>(Yp, pos, w, T, k, P, static_cast<__nv_bfloat16*>(Y));
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tffn
