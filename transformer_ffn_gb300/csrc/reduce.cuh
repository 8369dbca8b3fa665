// reduce.cuh -- the reduce-add form of the fused FFN, the kernel that
// "Kernel fusion and tensor parallelism", section "Step 1" describes.
//
// A task is one tile H[i, j] (band i of 256 rows, hidden tile j of 256
// columns).  The CTA pair computes it (X[i, :] W1[:, j], + b1, act1, bf16)
// into shared memory -- H never reaches global memory -- and multiplies it at
// once by every tile of row j of W2:  Y[i, k] += H[i, j] W2[j, k] for all k
// (the page's block-matrix product).  Each product leaves tensor memory through
// shared memory as asynchronous tile reductions (cp.reduce.async.bulk.tensor,
// fp32 add) into an fp32 copy of Y in the workspace.  An epilogue warp issues
// the reduction of one chunk while it loads the next, and the accumulator is
// double-buffered, so the next product's MMAs run while the reductions drain
// (the page's ping-pong between products and reductions).  A counter per
// 32-row strip of each Y tile counts the contributions (one per hidden tile);
// the warp that makes the last one reads the strip back, adds b2, applies act2
// and writes bf16 Y: the page's per-tile counter, with the final step taken
// by the last contributor as in Stream-K, which the page cites for this
// bookkeeping.
//
// Compared with the engine in engine.cuh (which sums over the hidden
// dimension in tensor memory and keeps H in L2), this form moves a 256-row
// fp32 partial of Y through L2 for every (H tile, W2 tile) pair, and its
// result depends on the order in which the reductions land (fp32 addition is
// not associative), so runs are not bit-reproducible.
//
// CTA layout (224 threads, clusters of two CTAs on two SMs, as the engine):
//   warp 0      A loader: the leader takes tickets and publishes tasks; each
//               CTA loads its 128 X rows per GEMM1 stage (a product stage
//               needs no A: A is the H tile in shared memory).
//   warp 6      B loader: W1 columns for GEMM1, then the W2 tiles of row j.
//   warp 1      leader: the pair MMAs (GEMM1 from the stages, products with A
//               from the H tile) and their commits.
//   warps 2..5  epilogue: H tile into shared memory; product chunks into the
//               staging buffers and out as tile reductions; counters; the
//               last contributor's b2 / act2 / bf16 pass.
// Shared memory per CTA: 4 stages x 32 KiB, the H tile (128 rows x 256
// hidden columns, K-major, 128-byte swizzle: 4 blocks of 16 KiB), two 4 KiB
// staging buffers per epilogue warp, the barrier block.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "engine.cuh"
#include "reduce_params.cuh"

namespace tffn {
namespace reduce {

// ----------------------------------------------------------------- producer
__device__ void run_producer(const Params& p, Aux& aux, uint8_t* smem, const WaitCtx& w, uint32_t rank)
{
    const int nk1 = (p.N + BK - 1) / BK;
    const int nk2 = p.n_p * (BN / BK);
    const int64_t total = static_cast<int64_t>(p.m_blocks) * p.n_h;
    uint32_t stage = 0, phase = 0;
    engine::Ring ring;
    int32_t last_phase[STAGES];
    for (int s = 0; s < STAGES; ++s)
        last_phase[s] = -1;

    for (;;) {
        int4 task;
        if (rank == 0) {
            const uint32_t t = atomicAdd(&p.ctrl->ticket, 1u);
            // Hidden-tile-major order: the bands in flight share the W1 / W2
            // tiles of a few hidden tiles.
            task = static_cast<int64_t>(t) < total
                       ? make_int4(0, static_cast<int32_t>(t % p.m_blocks), static_cast<int32_t>(t / p.m_blocks), 0)
                       : make_int4(-1, 0, 0, 0);
            if (!wait_mbar_cl(w, ptx::smem_u32(&aux.task_empty[ring.slot]), ring.phase ^ 1u, SITE_TASK_EMPTY))
                break;
            engine::publish_task(aux, ring, task);
        } else if (!engine::read_task(aux, w, ring, rank, false, 0, task)) {
            break;
        }
        if (task.x < 0)
            break;

        const int32_t row0 = task.y * BM + static_cast<int32_t>(rank) * BM_CTA;
        bool ok = true;
        for (int kb = 0; kb < nk1 + nk2; ++kb) {
            ok = wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY);
            if (!ok)
                break;
            const uint32_t fb_local = ptx::smem_u32(&aux.full[stage]);
            if (kb < nk1) {
                if (rank == 0)
                    ptx::mbar_arrive_expect_tx(fb_local, 2 * STAGE_BYTES);
                ptx::tma_load_2d_pair(ptx::smem_u32(smem + stage * STAGE_BYTES), &p.map_x, ptx::mapa(fb_local, 0),
                                      kb * BK, row0);
            } else if (rank == 0) {
                ptx::mbar_arrive_expect_tx(fb_local, 2 * B_STAGE_BYTES);   // W2 only: A is the H tile
            }
            last_phase[stage] = static_cast<int32_t>(phase);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok)
            break;
    }
    if (rank == 0)
        for (int s = 0; s < STAGES; ++s)
            if (last_phase[s] >= 0)
                engine::wait_own(w, ptx::smem_u32(&aux.full[s]), static_cast<uint32_t>(last_phase[s]));
}

// ---------------------------------------------------------------- B loader
__device__ void run_b_loader(const Params& p, Aux& aux, uint8_t* smem, const WaitCtx& w, uint32_t rank)
{
    const int nk1 = (p.N + BK - 1) / BK;
    const int nb = nk1 + p.n_p * (BN / BK);
    uint32_t stage = 0, phase = 0;
    engine::Ring ring;
    for (;;) {
        int4 task;
        if (!engine::read_task(aux, w, ring, rank, false, 0, task))
            break;
        if (task.x < 0)
            break;
        for (int kb = 0; kb < nb; ++kb) {
            if (!wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY))
                return;
            const uint32_t fb = ptx::mapa(ptx::smem_u32(&aux.full[stage]), 0);   // the leader's barrier
            const uint32_t sb = ptx::smem_u32(smem + stage * STAGE_BYTES) + A_STAGE_BYTES;
            const CUtensorMap* mb;
            int32_t col0, krow;
            if (kb < nk1) {           // W1[:, tile j]
                mb = &p.map_w1;
                col0 = task.z * BN + static_cast<int32_t>(rank) * BN_CTA;
                krow = kb * BK;
            } else {                  // W2[tile j rows, tile k]
                const int q = kb - nk1;
                mb = &p.map_w2;
                col0 = (q / (BN / BK)) * BN + static_cast<int32_t>(rank) * BN_CTA;
                krow = task.z * BN + (q % (BN / BK)) * BK;
            }
            if (p.b3d) {
                ptx::tma_load_3d_pair(sb, mb, fb, 0, krow, col0 / 64);
            } else {
#pragma unroll
                for (int i = 0; i < BN_CTA / 64; ++i)
                    ptx::tma_load_2d_pair(sb + i * B_BOX_BYTES, mb, fb, col0 + i * 64, krow);
            }
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// ------------------------------------------------------------- leader: MMA
__device__ void run_mma(const Params& p, Aux& aux, uint8_t* smem, const WaitCtx& w, uint32_t tmem_base)
{
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, 0, 1);
    const int nk1 = (p.N + BK - 1) / BK;
    const uint32_t h_base = ptx::smem_u32(smem + OFF_H);
    uint32_t stage = 0, phase = 0, iter = 0, htask = 0;
    engine::Ring ring;
    bool ok = true;
    for (;;) {
        int4 task;
        if (!engine::read_task(aux, w, ring, 0, false, 0, task))
            break;
        if (task.x < 0)
            break;
        // t = 0: GEMM1 into an accumulator; t = 1..n_p: the H tile times W2
        // tile t-1, with A read from the H tile in shared memory.
        for (int t = 0; t <= p.n_p; ++t) {
            const uint32_t acc = iter & 1u;
            const uint32_t acc_phase = (iter >> 1) & 1u;
            if (t == 1) {
                ok = wait_mbar_cl(w, ptx::smem_u32(&aux.h_full), htask & 1u, SITE_H_SMEM);
                if (!ok)
                    break;
            }
            ok = wait_mbar_cl(w, ptx::smem_u32(&aux.tmem_empty[acc]), acc_phase ^ 1u, SITE_TMEM_EMPTY);
            if (!ok)
                break;
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            const int nkb = t == 0 ? nk1 : BN / BK;
            for (int kb = 0; kb < nkb; ++kb) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.full[stage]), phase, SITE_SMEM_FULL);
                if (!ok)
                    break;
                ptx::tc_fence_after();
                const uint32_t sa = ptx::smem_u32(smem + stage * STAGE_BYTES);
                // A: K-major rows of 128 B, 8-row groups 1 KiB apart (a TMA
                // stage, or one 64-column block of the H tile).
                const uint64_t adesc = ptx::sdesc_sw128(t == 0 ? sa : h_base + kb * H_BLOCK_BYTES, 16, 1024);
                const uint64_t bdesc = ptx::sdesc_sw128(sa + A_STAGE_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    ptx::umma_bf16_pair(d_tmem, adesc + static_cast<uint64_t>((k * 32) >> 4),
                                        bdesc + static_cast<uint64_t>((k * 2048) >> 4), idesc,
                                        (kb > 0 || k > 0) ? 1u : 0u);
                ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.empty[stage]), 0x3);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.tmem_full[acc]), 0x3);
            ++iter;
        }
        if (!ok)
            break;
        ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.h_empty), 0x3);   // every reader of the H tile is done
        ++htask;
    }
    ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.drain), 0x1);
    engine::wait_own(w, ptx::smem_u32(&aux.drain), 0u);
}

// ---------------------------------------------------------------- epilogue
// GEMM1 accumulator -> H tile in shared memory, in the layout a TMA copy of a
// {64, 128} box with 128-byte swizzle would produce: block c/2 holds hidden
// columns [64*(c/2), +64); row r occupies 128 B at r*128; its 16-byte chunk q
// sits at position q ^ (r % 8).  Columns past O are zero.
template <int ACT>
__device__ __forceinline__ void h_tile(const Params& p, uint32_t taddr, int32_t j, uint32_t h_base, uint32_t row_local)
{
    for (int c = 0; c < CHUNKS; ++c) {
        uint32_t r[32];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
        ptx::tmem_ld_wait();
        const int32_t col = j * BN + c * 32;
        uint32_t packed[16];
#pragma unroll
        for (int g = 0; g < 4; ++g) {   // 8 columns per group; O % 8 == 0, so a group is all in or all out
            const bool in = col + g * 8 < p.O;
            uint4 bu = make_uint4(0u, 0u, 0u, 0u);
            if (in && p.b1 != nullptr)
                bu = __ldg(reinterpret_cast<const uint4*>(p.b1 + col + g * 8));
            const float b[8] = {bf16_lo(bu.x), bf16_hi(bu.x), bf16_lo(bu.y), bf16_hi(bu.y),
                                bf16_lo(bu.z), bf16_hi(bu.z), bf16_lo(bu.w), bf16_hi(bu.w)};
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[e] = in ? act_apply(ACT, __uint_as_float(r[g * 8 + e]) + b[e]) : 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                packed[g * 4 + e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
        }
        const uint32_t blk = h_base + (c >> 1) * H_BLOCK_BYTES + row_local * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t pos = ((static_cast<uint32_t>((c & 1) * 4 + q)) ^ (row_local & 7u)) * 16u;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(blk + pos), "r"(packed[q * 4]),
                         "r"(packed[q * 4 + 1]), "r"(packed[q * 4 + 2]), "r"(packed[q * 4 + 3])
                         : "memory");
        }
    }
}

// The last contributor's pass over its strip: row `row`, columns
// [col0, col0 + ncol) of the fp32 accumulator -> + b2, act2, bf16 Y.
template <int ACT>
__device__ __forceinline__ void finish_row(const Params& p, int64_t row, int32_t col0, int32_t ncol)
{
    const float* src = p.acc + row * p.P + col0;
    __nv_bfloat16* dst = p.Y + row * p.P + col0;
    for (int32_t c = 0; c < ncol; c += 8) {
        // the other SMs' reductions landed in L2: read at L2, not L1
        const float4 a = __ldcg(reinterpret_cast<const float4*>(src + c));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(src + c + 4));
        uint4 bu = make_uint4(0u, 0u, 0u, 0u);
        if (p.b2 != nullptr)
            bu = __ldg(reinterpret_cast<const uint4*>(p.b2 + col0 + c));
        const uint4 o = make_uint4(
            pack_bf16x2(act_apply(ACT, a.x + bf16_lo(bu.x)), act_apply(ACT, a.y + bf16_hi(bu.x))),
            pack_bf16x2(act_apply(ACT, a.z + bf16_lo(bu.y)), act_apply(ACT, a.w + bf16_hi(bu.y))),
            pack_bf16x2(act_apply(ACT, b.x + bf16_lo(bu.z)), act_apply(ACT, b.y + bf16_hi(bu.z))),
            pack_bf16x2(act_apply(ACT, b.z + bf16_lo(bu.w)), act_apply(ACT, b.w + bf16_hi(bu.w))));
        *reinterpret_cast<uint4*>(dst + c) = o;
    }
}

// Count one contribution to the warp's strip of Y tile (i, k), after this
// warp's reductions into it have completed; the last one finishes the strip.
__device__ __noinline__ void contribute(const Params& p, int32_t i, int32_t k, uint32_t rank, uint32_t quad,
                                        int lane)
{
    uint32_t* ctr = p.counters + (static_cast<int64_t>(i) * p.n_p + k) * COUNTERS_PER_TILE + rank * EPI_WARPS + quad;
    uint32_t last = 0;
    if (lane == 0) {
        ptx::fence_proxy_async_global();   // the completed tile reductions before the release below
        __threadfence();
        last = atomicAdd(ctr, 1u) == static_cast<uint32_t>(p.n_h - 1) ? 1u : 0u;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last)
        return;
    __threadfence();   // every contribution counted before ours is visible
    const int64_t row = static_cast<int64_t>(i) * BM + rank * BM_CTA + quad * 32 + lane;
    if (row >= p.M)
        return;
    const int32_t col0 = k * BN;
    const int32_t ncol = p.P - col0 < BN ? p.P - col0 : BN;
    switch (p.act2) {
    case TFFN_ACT_GELU_TANH: finish_row<TFFN_ACT_GELU_TANH>(p, row, col0, ncol); break;
    case TFFN_ACT_SILU: finish_row<TFFN_ACT_SILU>(p, row, col0, ncol); break;
    case TFFN_ACT_RELU: finish_row<TFFN_ACT_RELU>(p, row, col0, ncol); break;
    default: finish_row<TFFN_ACT_NONE>(p, row, col0, ncol); break;
    }
}

__device__ void run_epilogue(const Params& p, Aux& aux, uint8_t* smem, const WaitCtx& w, uint32_t tmem_base,
                             uint32_t rank, int warp, int lane)
{
    const uint32_t quad = static_cast<uint32_t>(warp & 3);   // TMEM lanes [32*quad, 32*quad+32)
    const uint32_t row_local = quad * 32 + static_cast<uint32_t>(lane);
    const uint32_t h_base = ptx::smem_u32(smem + OFF_H);
    const uint32_t stg = ptx::smem_u32(smem + OFF_STG) + static_cast<uint32_t>(warp - 2) * STG_BUFS * STG_BYTES;
    uint32_t iter = 0, htask = 0, nred = 0;
    int32_t pend_i = -1, pend_k = 0;   // strip whose contribution waits for its reductions
    bool failed = false;
    engine::Ring ring;
    for (;;) {
        int4 task;
        if (!engine::read_task(aux, w, ring, rank, true, lane, task))
            break;
        if (task.x < 0)
            break;
        const int32_t i = task.y, j = task.z;

        // ---- GEMM1 -> H tile in shared memory
        {
            const uint32_t acc = iter & 1u;
            const uint32_t acc_phase = (iter >> 1) & 1u;
            if (!wait_mbar(w, ptx::smem_u32(&aux.tmem_full[acc]), acc_phase, SITE_TMEM_FULL) ||
                !wait_mbar(w, ptx::smem_u32(&aux.h_empty), (htask & 1u) ^ 1u, SITE_H_FREE)) {
                failed = true;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + acc * BN;
            switch (p.act1) {
            case TFFN_ACT_GELU_TANH: h_tile<TFFN_ACT_GELU_TANH>(p, taddr, j, h_base, row_local); break;
            case TFFN_ACT_SILU: h_tile<TFFN_ACT_SILU>(p, taddr, j, h_base, row_local); break;
            case TFFN_ACT_RELU: h_tile<TFFN_ACT_RELU>(p, taddr, j, h_base, row_local); break;
            default: h_tile<TFFN_ACT_NONE>(p, taddr, j, h_base, row_local); break;
            }
            ptx::fence_proxy_async_smem();   // the MMAs (async proxy) read what the threads wrote
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                engine::arrive_on_leader(ptx::smem_u32(&aux.tmem_empty[acc]), rank);
                engine::arrive_on_leader(ptx::smem_u32(&aux.h_full), rank);
            }
            ++iter;
            ++htask;
        }

        // ---- H tile x W2 tiles of row j -> reductions into the Y accumulator
        const int32_t ry = i * BM + static_cast<int32_t>(rank) * BM_CTA + static_cast<int32_t>(quad) * 32;
        for (int32_t k = 0; k < p.n_p; ++k) {
            const uint32_t acc = iter & 1u;
            const uint32_t acc_phase = (iter >> 1) & 1u;
            if (!wait_mbar(w, ptx::smem_u32(&aux.tmem_full[acc]), acc_phase, SITE_TMEM_FULL)) {
                failed = true;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + acc * BN;
            const int32_t col0 = k * BN;
            const int nch = p.P - col0 >= BN ? CHUNKS : (p.P - col0 + 31) / 32;
            for (int c = 0; c < nch; ++c) {
                uint32_t r[32];
                __syncwarp();
                ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
                ptx::tmem_ld_wait();
                const uint32_t buf = stg + (nred & 1u) * STG_BYTES;
                if (nred >= STG_BUFS && lane == 0)
                    ptx::bulk_wait_group_read<STG_BUFS - 1>();   // the buffer's last reduction has read it
                __syncwarp();
                // row `lane` of the box: 128 B; 16-byte chunk q at position q ^ (lane % 8)
                const uint32_t rowa = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t pos = (static_cast<uint32_t>(q) ^ (static_cast<uint32_t>(lane) & 7u)) * 16u;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rowa + pos), "r"(r[q * 4]),
                                 "r"(r[q * 4 + 1]), "r"(r[q * 4 + 2]), "r"(r[q * 4 + 3])
                                 : "memory");
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_reduce_add_2d(&p.map_acc, buf, col0 + c * 32, ry);
                    ptx::bulk_commit_group();
                }
                ++nred;
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                engine::arrive_on_leader(ptx::smem_u32(&aux.tmem_empty[acc]), rank);
            ++iter;
            // The previous strip's reductions are complete once no more than
            // this tile's groups are outstanding.
            if (pend_i >= 0) {
                if (lane == 0) {
                    if (nch == CHUNKS)
                        ptx::bulk_wait_group<CHUNKS>();
                    else
                        ptx::bulk_wait_group<0>();
                }
                __syncwarp();
                contribute(p, pend_i, pend_k, rank, quad, lane);
            }
            pend_i = i;
            pend_k = k;
        }
        if (failed)
            break;
    }
    // Every reduction this warp issued completes before the CTA leaves (its
    // staging buffers are read until then).
    if (lane == 0)
        ptx::bulk_wait_group<0>();
    __syncwarp();
    if (!failed && pend_i >= 0 && !*reinterpret_cast<volatile uint32_t*>(w.abort))
        contribute(p, pend_i, pend_k, rank, quad, lane);
}

// ------------------------------------------------------------------- kernel
__global__ void __launch_bounds__(NUM_THREADS, 1) reduce_kernel(const __grid_constant__ Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Aux& aux = *reinterpret_cast<Aux*>(smem + OFF_AUX);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = ptx::cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_u32(&aux.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_u32(&aux.tmem_full[a]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.tmem_empty[a]), 2 * EPI_WARPS);
        }
        ptx::mbar_init(ptx::smem_u32(&aux.h_full), 2 * EPI_WARPS);
        ptx::mbar_init(ptx::smem_u32(&aux.h_empty), 1);
        for (int s = 0; s < TASK_SLOTS; ++s) {
            ptx::mbar_init(ptx::smem_u32(&aux.task_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.task_empty[s]), TASK_CONSUMERS);
        }
        ptx::mbar_init(ptx::smem_u32(&aux.drain), 1);
        aux.abort = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&p.map_x);
        ptx::prefetch_tmap(&p.map_w1);
        ptx::prefetch_tmap(&p.map_w2);
        ptx::prefetch_tmap(&p.map_acc);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(&aux.tmem_base), TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem_base = aux.tmem_base;

    const WaitCtx w{&aux.abort, p.ctrl, p.wait_limit_ns, ptx::mapa(ptx::smem_u32(&aux.abort), rank ^ 1u)};
    if (warp == 0) {
        if (lane == 0)
            run_producer(p, aux, smem, w, rank);
    } else if (warp == B_LOADER_WARP) {
        if (lane == 0)
            run_b_loader(p, aux, smem, w, rank);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0)
            run_mma(p, aux, smem, w, tmem_base);
    } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
        run_epilogue(p, aux, smem, w, tmem_base, rank, warp, lane);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();   // the leader's MMAs read the peer's shared memory
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&p.ctrl->done, 1u) == gridDim.x - 1) {
            p.ctrl->ticket = 0u;
            p.ctrl->done = 0u;
            __threadfence();
        }
    }
}

// ===================================================================== b2b
// Back-to-back form for small FFNs (H on chip, BOLT-style, as "Kernel fusion
// and tensor parallelism", section "Step 1" describes back-to-back GEMM
// kernels): a task is (band i, Y tile k).  The pair walks the hidden tiles
// j: GEMM1 tile j into one accumulator, + b1 and act1 into the H tile in
// shared memory, then the product H[i, j] W2[j, k] added into a second
// accumulator that lives for the whole task.  After the last hidden tile the
// second accumulator holds Y[i, k] over the full hidden dimension: + b2, act2,
// bf16, stored.  No H in global memory, no flags, no reductions; the price is
// that each task recomputes its band's H (once per Y tile of the band), so
// the form suits FFNs whose Y has few column tiles.
//
// Tensor memory: columns [0, 256) hold the GEMM1 accumulator, [256, 512) the
// Y accumulator.  Warp roles and shared memory as the reduce-add form (the
// staging buffers are unused).

struct B2BAux {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t g_full;     // GEMM1 accumulator ready (multicast commit)
    uint64_t g_empty;    // leader: the pair's eight epilogue warps drained it
    uint64_t y_full;     // Y accumulator complete (multicast commit)
    uint64_t y_empty;    // leader: drained
    uint64_t h_full;     // leader: H tile written by the pair's eight epilogue warps
    uint64_t h_empty;    // the MMAs reading the H tile are done (multicast commit)
    uint64_t task_full[TASK_SLOTS];
    uint64_t task_empty[TASK_SLOTS];
    uint64_t drain;
    int4 task[TASK_SLOTS];
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(B2BAux) <= AUX_BYTES, "aux block fits");

__device__ void b2b_producer(const Params& p, B2BAux& aux, uint8_t* smem, const WaitCtx& w, uint32_t rank)
{
    const int nk1 = (p.N + BK - 1) / BK;
    const int64_t total = static_cast<int64_t>(p.m_blocks) * p.n_p;
    uint32_t stage = 0, phase = 0;
    engine::Ring ring;
    int32_t last_phase[STAGES];
    for (int s = 0; s < STAGES; ++s)
        last_phase[s] = -1;
    for (;;) {
        int4 task;
        if (rank == 0) {
            const uint32_t t = atomicAdd(&p.ctrl->ticket, 1u);
            task = static_cast<int64_t>(t) < total
                       ? make_int4(0, static_cast<int32_t>(t % p.m_blocks), static_cast<int32_t>(t / p.m_blocks), 0)
                       : make_int4(-1, 0, 0, 0);
            if (!wait_mbar_cl(w, ptx::smem_u32(&aux.task_empty[ring.slot]), ring.phase ^ 1u, SITE_TASK_EMPTY))
                break;
            engine::publish_task(aux, ring, task);
        } else if (!engine::read_task(aux, w, ring, rank, false, 0, task)) {
            break;
        }
        if (task.x < 0)
            break;
        const int32_t row0 = task.y * BM + static_cast<int32_t>(rank) * BM_CTA;
        bool ok = true;
        for (int32_t j = 0; j < p.n_h && ok; ++j) {
            for (int kb = 0; kb < nk1 + BN / BK; ++kb) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY);
                if (!ok)
                    break;
                const uint32_t fb_local = ptx::smem_u32(&aux.full[stage]);
                if (kb < nk1) {
                    if (rank == 0)
                        ptx::mbar_arrive_expect_tx(fb_local, 2 * STAGE_BYTES);
                    ptx::tma_load_2d_pair(ptx::smem_u32(smem + stage * STAGE_BYTES), &p.map_x,
                                          ptx::mapa(fb_local, 0), kb * BK, row0);
                } else if (rank == 0) {
                    ptx::mbar_arrive_expect_tx(fb_local, 2 * B_STAGE_BYTES);   // W2 only: A is the H tile
                }
                last_phase[stage] = static_cast<int32_t>(phase);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok)
            break;
    }
    if (rank == 0)
        for (int s = 0; s < STAGES; ++s)
            if (last_phase[s] >= 0)
                engine::wait_own(w, ptx::smem_u32(&aux.full[s]), static_cast<uint32_t>(last_phase[s]));
}

__device__ void b2b_b_loader(const Params& p, B2BAux& aux, uint8_t* smem, const WaitCtx& w, uint32_t rank)
{
    const int nk1 = (p.N + BK - 1) / BK;
    uint32_t stage = 0, phase = 0;
    engine::Ring ring;
    for (;;) {
        int4 task;
        if (!engine::read_task(aux, w, ring, rank, false, 0, task))
            break;
        if (task.x < 0)
            break;
        for (int32_t j = 0; j < p.n_h; ++j) {
            for (int kb = 0; kb < nk1 + BN / BK; ++kb) {
                if (!wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY))
                    return;
                const uint32_t fb = ptx::mapa(ptx::smem_u32(&aux.full[stage]), 0);
                const uint32_t sb = ptx::smem_u32(smem + stage * STAGE_BYTES) + A_STAGE_BYTES;
                const CUtensorMap* mb;
                int32_t col0, krow;
                if (kb < nk1) {           // W1[:, tile j]
                    mb = &p.map_w1;
                    col0 = j * BN + static_cast<int32_t>(rank) * BN_CTA;
                    krow = kb * BK;
                } else {                  // W2[tile j rows, tile k]
                    mb = &p.map_w2;
                    col0 = task.z * BN + static_cast<int32_t>(rank) * BN_CTA;
                    krow = j * BN + (kb - nk1) * BK;
                }
                if (p.b3d) {
                    ptx::tma_load_3d_pair(sb, mb, fb, 0, krow, col0 / 64);
                } else {
#pragma unroll
                    for (int i = 0; i < BN_CTA / 64; ++i)
                        ptx::tma_load_2d_pair(sb + i * B_BOX_BYTES, mb, fb, col0 + i * 64, krow);
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
}

__device__ void b2b_mma(const Params& p, B2BAux& aux, uint8_t* smem, const WaitCtx& w, uint32_t tmem_base)
{
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, 0, 1);
    const int nk1 = (p.N + BK - 1) / BK;
    const uint32_t h_base = ptx::smem_u32(smem + OFF_H);
    const uint32_t g_tmem = tmem_base;
    const uint32_t y_tmem = tmem_base + BN;
    uint32_t stage = 0, phase = 0, gi = 0, hi = 0, yi = 0;
    engine::Ring ring;
    bool ok = true;
    for (;;) {
        int4 task;
        if (!engine::read_task(aux, w, ring, 0, false, 0, task))
            break;
        if (task.x < 0)
            break;
        for (int32_t j = 0; j < p.n_h && ok; ++j) {
            // GEMM1 tile j
            ok = wait_mbar_cl(w, ptx::smem_u32(&aux.g_empty), (gi & 1u) ^ 1u, SITE_TMEM_EMPTY);
            if (!ok)
                break;
            ptx::tc_fence_after();
            for (int kb = 0; kb < nk1; ++kb) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.full[stage]), phase, SITE_SMEM_FULL);
                if (!ok)
                    break;
                ptx::tc_fence_after();
                const uint32_t sa = ptx::smem_u32(smem + stage * STAGE_BYTES);
                const uint64_t adesc = ptx::sdesc_sw128(sa, 16, 1024);
                const uint64_t bdesc = ptx::sdesc_sw128(sa + A_STAGE_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    ptx::umma_bf16_pair(g_tmem, adesc + static_cast<uint64_t>((k * 32) >> 4),
                                        bdesc + static_cast<uint64_t>((k * 2048) >> 4), idesc,
                                        (kb > 0 || k > 0) ? 1u : 0u);
                ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.empty[stage]), 0x3);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.g_full), 0x3);
            ++gi;
            // the product with W2[j, k], accumulated over j
            ok = wait_mbar_cl(w, ptx::smem_u32(&aux.h_full), hi & 1u, SITE_H_SMEM);
            if (ok && j == 0)
                ok = wait_mbar_cl(w, ptx::smem_u32(&aux.y_empty), (yi & 1u) ^ 1u, SITE_TMEM_EMPTY);
            if (!ok)
                break;
            ptx::tc_fence_after();
            for (int kb = 0; kb < BN / BK; ++kb) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.full[stage]), phase, SITE_SMEM_FULL);
                if (!ok)
                    break;
                ptx::tc_fence_after();
                const uint32_t sa = ptx::smem_u32(smem + stage * STAGE_BYTES);
                const uint64_t adesc = ptx::sdesc_sw128(h_base + kb * H_BLOCK_BYTES, 16, 1024);
                const uint64_t bdesc = ptx::sdesc_sw128(sa + A_STAGE_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    ptx::umma_bf16_pair(y_tmem, adesc + static_cast<uint64_t>((k * 32) >> 4),
                                        bdesc + static_cast<uint64_t>((k * 2048) >> 4), idesc,
                                        (j > 0 || kb > 0 || k > 0) ? 1u : 0u);
                ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.empty[stage]), 0x3);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.h_empty), 0x3);
            ++hi;
        }
        if (!ok)
            break;
        ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.y_full), 0x3);
        ++yi;
    }
    ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.drain), 0x1);
    engine::wait_own(w, ptx::smem_u32(&aux.drain), 0u);
}

// Y accumulator -> + b2, act2, bf16 Y for the thread's row.
template <int ACT>
__device__ __forceinline__ void y_tile(const Params& p, uint32_t taddr, int32_t col0, int64_t row)
{
    const int nch = p.P - col0 >= BN ? CHUNKS : (p.P - col0 + 31) / 32;
    for (int c = 0; c < nch; ++c) {
        uint32_t r[32];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
        ptx::tmem_ld_wait();
        if (row >= p.M)
            continue;
        const int32_t col = col0 + c * 32;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (col + g * 8 >= p.P)
                break;
            uint4 bu = make_uint4(0u, 0u, 0u, 0u);
            if (p.b2 != nullptr)
                bu = __ldg(reinterpret_cast<const uint4*>(p.b2 + col + g * 8));
            const float* a = reinterpret_cast<const float*>(r + g * 8);
            const uint4 o = make_uint4(
                pack_bf16x2(act_apply(ACT, a[0] + bf16_lo(bu.x)), act_apply(ACT, a[1] + bf16_hi(bu.x))),
                pack_bf16x2(act_apply(ACT, a[2] + bf16_lo(bu.y)), act_apply(ACT, a[3] + bf16_hi(bu.y))),
                pack_bf16x2(act_apply(ACT, a[4] + bf16_lo(bu.z)), act_apply(ACT, a[5] + bf16_hi(bu.z))),
                pack_bf16x2(act_apply(ACT, a[6] + bf16_lo(bu.w)), act_apply(ACT, a[7] + bf16_hi(bu.w))));
            *reinterpret_cast<uint4*>(p.Y + row * p.P + col + g * 8) = o;
        }
    }
}

__device__ void b2b_epilogue(const Params& p, B2BAux& aux, uint8_t* smem, const WaitCtx& w, uint32_t tmem_base,
                             uint32_t rank, int warp, int lane)
{
    const uint32_t quad = static_cast<uint32_t>(warp & 3);
    const uint32_t row_local = quad * 32 + static_cast<uint32_t>(lane);
    const uint32_t h_base = ptx::smem_u32(smem + OFF_H);
    const uint32_t lanes = (quad * 32u) << 16;
    uint32_t gi = 0, hi = 0, yi = 0;
    engine::Ring ring;
    for (;;) {
        int4 task;
        if (!engine::read_task(aux, w, ring, rank, true, lane, task))
            break;
        if (task.x < 0)
            break;
        bool ok = true;
        for (int32_t j = 0; j < p.n_h; ++j) {
            ok = wait_mbar(w, ptx::smem_u32(&aux.g_full), gi & 1u, SITE_TMEM_FULL) &&
                 wait_mbar(w, ptx::smem_u32(&aux.h_empty), (hi & 1u) ^ 1u, SITE_H_FREE);
            if (!ok)
                break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + lanes;
            switch (p.act1) {
            case TFFN_ACT_GELU_TANH: h_tile<TFFN_ACT_GELU_TANH>(p, taddr, j, h_base, row_local); break;
            case TFFN_ACT_SILU: h_tile<TFFN_ACT_SILU>(p, taddr, j, h_base, row_local); break;
            case TFFN_ACT_RELU: h_tile<TFFN_ACT_RELU>(p, taddr, j, h_base, row_local); break;
            default: h_tile<TFFN_ACT_NONE>(p, taddr, j, h_base, row_local); break;
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                engine::arrive_on_leader(ptx::smem_u32(&aux.g_empty), rank);
                engine::arrive_on_leader(ptx::smem_u32(&aux.h_full), rank);
            }
            ++gi;
            ++hi;
        }
        if (!ok || !wait_mbar(w, ptx::smem_u32(&aux.y_full), yi & 1u, SITE_TMEM_FULL))
            break;
        ptx::tc_fence_after();
        const uint32_t taddr = tmem_base + lanes + BN;
        const int64_t row = static_cast<int64_t>(task.y) * BM + rank * BM_CTA + row_local;
        const int32_t col0 = task.z * BN;
        switch (p.act2) {
        case TFFN_ACT_GELU_TANH: y_tile<TFFN_ACT_GELU_TANH>(p, taddr, col0, row); break;
        case TFFN_ACT_SILU: y_tile<TFFN_ACT_SILU>(p, taddr, col0, row); break;
        case TFFN_ACT_RELU: y_tile<TFFN_ACT_RELU>(p, taddr, col0, row); break;
        default: y_tile<TFFN_ACT_NONE>(p, taddr, col0, row); break;
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0)
            engine::arrive_on_leader(ptx::smem_u32(&aux.y_empty), rank);
        ++yi;
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) b2b_kernel(const __grid_constant__ Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    B2BAux& aux = *reinterpret_cast<B2BAux*>(smem + OFF_AUX);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = ptx::cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_u32(&aux.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&aux.g_full), 1);
        ptx::mbar_init(ptx::smem_u32(&aux.g_empty), 2 * EPI_WARPS);
        ptx::mbar_init(ptx::smem_u32(&aux.y_full), 1);
        ptx::mbar_init(ptx::smem_u32(&aux.y_empty), 2 * EPI_WARPS);
        ptx::mbar_init(ptx::smem_u32(&aux.h_full), 2 * EPI_WARPS);
        ptx::mbar_init(ptx::smem_u32(&aux.h_empty), 1);
        for (int s = 0; s < TASK_SLOTS; ++s) {
            ptx::mbar_init(ptx::smem_u32(&aux.task_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.task_empty[s]), TASK_CONSUMERS);
        }
        ptx::mbar_init(ptx::smem_u32(&aux.drain), 1);
        aux.abort = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&p.map_x);
        ptx::prefetch_tmap(&p.map_w1);
        ptx::prefetch_tmap(&p.map_w2);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(&aux.tmem_base), TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = aux.tmem_base;

    const WaitCtx w{&aux.abort, p.ctrl, p.wait_limit_ns, ptx::mapa(ptx::smem_u32(&aux.abort), rank ^ 1u)};
    if (warp == 0) {
        if (lane == 0)
            b2b_producer(p, aux, smem, w, rank);
    } else if (warp == B_LOADER_WARP) {
        if (lane == 0)
            b2b_b_loader(p, aux, smem, w, rank);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0)
            b2b_mma(p, aux, smem, w, tmem_base);
    } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
        b2b_epilogue(p, aux, smem, w, tmem_base, rank, warp, lane);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&p.ctrl->done, 1u) == gridDim.x - 1) {
            p.ctrl->ticket = 0u;
            p.ctrl->done = 0u;
            __threadfence();
        }
    }
}

}  // namespace reduce
}  // namespace tffn
