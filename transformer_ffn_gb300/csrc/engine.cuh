// engine.cuh -- the persistent, warp-specialised 2-SM tcgen05 engine that runs
// the two GEMMs of the FFN (and of every expert of the MoE form) in one launch.
//
// What it computes ("Kernel fusion and tensor parallelism", section
// "Megatron-LM tensor parallelism", FFN equation; section "Step 1"):
//   layer 1 tile (band i, tile j):  H[i, j] = bf16(act1(X[i, :] W1[:, j] + b1[j]))
//   layer 2 tile (band i, tile k):  Y[i, k] = act2(H[i, :] W2[:, k] + b2[k])
// with fp32 accumulation in tensor memory.  A layer-1 tile publishes ready
// flags once its H tile is in global memory and counts itself in its band's
// tally; a layer-2 tile of the same band starts at once when the tally says
// the whole band is written, and otherwise waits on the flags chunk by chunk
// before its TMA loads read H, so H is consumed while the rest of H is still
// being produced (the page's per-tile flag, used here between the SMs of one
// GPU).
//
// Tiles are 256 x 256 and belong to a cluster of two CTAs on two SMs (a CTA
// pair): tcgen05.mma.cta_group::2 with M = 256 reads A's rows split between
// the pair (128 each) and B's columns split between the pair (128 each), and
// writes each CTA's tensor memory with its 128 rows x 256 columns.  Each CTA
// therefore streams only half of the B tile: 32 KiB per 64-deep k-stage per
// SM, six stages deep, beside 32 KiB of output staging buffers, the barrier
// block and one 1 KiB bias slice (all of a CTA's shared memory).
//
// CTA layout (224 threads, one CTA per SM, two CTAs per cluster):
//   warp 0      A loader.  The leader (cluster rank 0) takes tickets one
//               task ahead and publishes each task to both CTAs' task rings;
//               each A loader streams its CTA's A rows (and, for layer 2,
//               checks that H is ready first).
//   warp 6      B loader: streams the CTA's B columns, one TMA copy per stage
//               (a 3-D map covers both 64-column halves).  A and B copies are
//               issued by different warps because one warp issues bulk copies
//               one after the other; the B loader needs no flags and runs
//               ahead freely.  Every copy of the pair counts its bytes on the
//               leader's stage barrier (cta_group::2 copies).
//   warp 1      leader: issues the pair MMAs from one thread and commits
//               them to both CTAs' barriers (multicast).  Both CTAs: own the
//               CTA's tensor memory (512 columns = two accumulators of 128
//               lanes x 256 fp32 columns).
//   warps 2..5  epilogue: tcgen05.ld the CTA's accumulator (one TMEM lane
//               quadrant per warp, one row per thread), bias, activation,
//               round, write the rows into the warp's swizzled staging
//               buffer, TMA-store each 32-row box; the accumulator is
//               double-buffered so the epilogue of one tile overlaps the
//               main loop of the next.
//               The four warps share the tile's bias slice in shared memory
//               (each fetches a quarter before the accumulator wait).
//   warp 1 of the peer CTA has no role after the allocation.
//
// Operands: A (X or H) is row-major [rows x K]: K-major, 128-byte swizzle,
// boxes of 64 (K) x 128 (rows).  B (W1 or W2) is row-major [K x cols]: the
// columns are contiguous, so B is MN-major: two boxes of 64 (cols) x 64 (K)
// per CTA per stage, 128-byte swizzle.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "schedule.h"

namespace tffn {
namespace engine {

constexpr int BM = 256;                                   // rows of a pair tile (a band)
constexpr int BM_CTA = 128;                               // rows per CTA
constexpr int BN = 256;                                   // columns of a tile
constexpr int BN_CTA = 128;                               // B columns loaded per CTA
constexpr int BK = 64;
#ifndef TFFN_ENGINE_STAGES
#define TFFN_ENGINE_STAGES 6
#endif
constexpr int STAGES = TFFN_ENGINE_STAGES;              // 6 x 32 KiB, beside the output staging buffers
constexpr int A_STAGE_BYTES = BM_CTA * BK * 2;            // 16 KiB
constexpr int B_BOX_BYTES = 64 * BK * 2;                  // 8 KiB: 64 cols x 64 k
constexpr int B_STAGE_BYTES = BK * BN_CTA * 2;            // 16 KiB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int TASK_SLOTS = 4;
constexpr int NUM_THREADS = 224;
constexpr int B_LOADER_WARP = 6;
constexpr int EPI_WARPS = 4;
constexpr int FLAG_WORDS_PER_TILE = 2 * EPI_WARPS;        // one per epilogue warp of the pair
constexpr uint32_t TMEM_COLS = 512;
constexpr int AUX_BYTES = 1024;
constexpr int BIAS_BYTES = BN * 4;                        // the tile's fp32 bias, shared by the epilogue warps
// bf16 outputs leave through shared memory and TMA stores: each epilogue warp
// owns two 4 KiB buffers, each a 32-row x 64-column box in the 128-byte
// swizzled layout (per-thread row stores from the epilogue slowed the
// concurrent main loop's operand feed by 9-12 %).
constexpr int OUT_COLS = 64;
constexpr int OUT_BUF_BYTES = 32 * OUT_COLS * 2;          // 4 KiB
constexpr int OUT_BYTES = EPI_WARPS * 2 * OUT_BUF_BYTES;  // 32 KiB
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + AUX_BYTES + BIAS_BYTES + 1024;   // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
// Arrivals that free a task slot (counted on the leader): leader MMA thread,
// leader B loader, leader epilogue warps, peer A loader, peer B loader, peer
// epilogue warps.
constexpr uint32_t TASK_CONSUMERS = 1 + 1 + EPI_WARPS + 1 + 1 + EPI_WARPS;

// Per-layer arguments.
struct LayerArgs {
    int32_t K;          // reduction length (N for layer 1, O for layer 2)
    int32_t ncols;      // output columns (O, P)
    int32_t n_tiles;    // ceil(ncols / BN)
    int32_t act;        // tffn_act
    int32_t out_f32;    // 1: fp32 output, 0: bf16
    int32_t pad_;
    int64_t ld_out;     // output row stride in elements
    int64_t rows;       // rows of the output that are stored (later rows are skipped)
    void* out;
};

template <int MAX_E>
struct Params {
    CUtensorMap map_a[2];                      // layer-1 A (X), layer-2 A (H); box {64, 128}
    CUtensorMap map_out[2];                    // outputs H [rows x O], Y [rows x P] stored by TMA from the
                                               // epilogue: bf16 box {64, 32}; fp32 (MoE Y_perm) box {32, 32}
    CUtensorMap map_b[2][MAX_E];               // W1[e], W2[e]; b3d: {64, 64, 2} else {64, 64}
    const __nv_bfloat16* bias[2][MAX_E];       // b1[e], b2[e] (nullable)
    LayerArgs layer[2];
    int64_t m_blocks;                          // 256-row bands; < 0: read *m_blocks_dev
    const int32_t* m_blocks_dev;
    const int32_t* band_expert;                // expert of each band (NULL: expert 0)
    uint32_t* flags;                           // [m_blocks * n1 * 8] ready words
    // Per band and CTA rank: how many layer-1 epilogue warps of this launch
    // have published their rows of the band (n1 * EPI_WARPS: the CTA's whole
    // band of H is ready).  Zero when a launch starts; the last CTA out
    // zeroes it again.  NULL: layer-2 producers poll the per-tile flags only.
    uint32_t* band_count;                      // [m_blocks * 2]
    DevCtrl* ctrl;
    uint64_t wait_limit_ns;
    int32_t mode;                              // EngineMode
    int32_t group_m;
    int32_t skip_flag;                         // test fault injection, -1 = off
    int32_t b3d;                               // 1: map_b are 3-D {64 cols, K, cols/64} maps
    int32_t glu;                               // 1: layer 1 is gated, H = act(X W1) * (X W3)
    CUtensorMap map_b_lin[MAX_E];              // glu: W3[e], laid out like map_b[0][e]
    // MoE combine fused into the layer-2 epilogue (comb_cnt NULL: off; the
    // separate combine kernel runs instead).  row_entry[r] is the routing
    // entry t*k+s of grouped row r (-1 for a padding row, which is then not
    // stored); the last of a token's k rows to finish a Y column tile sums
    // the k expert outputs in slot order: Y[t] = sum_s w[t,s] Yp[pos[t,s]].
    const int32_t* row_entry;                  // [rows of the grouped layout]
    const int32_t* comb_pos;                   // [T * k] grouped row of each entry
    const float* comb_w;                       // [T * k] gate weights
    uint32_t* comb_cnt;                        // [T * n2] arrivals, reset by the last arriver
    __nv_bfloat16* comb_y;                     // Y [T x ncols of layer 2]
    int32_t comb_k;
};

// Hidden columns one layer-1 tile produces: a gated tile spends its 256
// accumulator columns on 128 gate and 128 linear columns of the same H slice.
template <int MAX_E>
__device__ __forceinline__ int32_t h_cols_per_tile(const Params<MAX_E>& p)
{
    return p.glu ? BN_CTA : BN;
}

// Everything in shared memory besides the stage ring (same offsets in both
// CTAs of a pair, which the cross-CTA addressing relies on).
struct Aux {
    uint64_t full[STAGES];          // leader: the TMA bytes of both CTAs (peer's copy unused)
    uint64_t empty[STAGES];         // MMA done with the stage (multicast commit)
    uint64_t tmem_full[2];          // accumulator ready (multicast commit)
    uint64_t tmem_empty[2];         // leader: eight epilogue warps of the pair drained it
    uint64_t task_full[TASK_SLOTS];
    uint64_t task_empty[TASK_SLOTS];    // leader only
    uint64_t drain;                 // leader: every MMA issued has completed
    uint64_t bias_ready;            // the four epilogue warps wrote the tile's bias slice
    uint64_t bias_free;             // the four epilogue warps are done reading it
    int4 task[TASK_SLOTS];
    uint32_t tmem_base;
    uint32_t abort;
    uint32_t epoch;                 // this launch's ready-flag value (control block's + 1)
};
static_assert(sizeof(Aux) <= AUX_BYTES, "aux block fits");

// Bounded wait that ignores the abort flag: used on the exit path to wait for
// this CTA's own copies and MMAs, which always complete.
__device__ __forceinline__ void wait_own(const WaitCtx& w, uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait_cluster(bar, parity)) {
        if (ptx::globaltimer() - t0 > w.limit_ns) {
            raise_error(w, static_cast<uint32_t>(TFFN_ERR_TIMEOUT), SITE_DRAIN, parity);
            return;
        }
    }
}

template <int MAX_E>
__device__ __forceinline__ int expert_of(const Params<MAX_E>& p, int band)
{
    if (MAX_E == 1 || p.band_expert == nullptr)
        return 0;
    return p.band_expert[band];
}

// Arrive on the leader's copy of a barrier (a local arrive on the leader).
__device__ __forceinline__ void arrive_on_leader(uint32_t bar, uint32_t rank)
{
    if (rank == 0)
        ptx::mbar_arrive(bar);
    else
        ptx::mbar_arrive_cluster(ptx::mapa(bar, 0));
}

// Position in the task ring.
struct Ring {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void advance()
    {
        if (++slot == TASK_SLOTS) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// Read the next task from this CTA's ring and free the slot on the leader
// (warp_wide: the whole warp waits, lane 0 arrives).  False on abort/timeout.
template <class AuxT>
__device__ __forceinline__ bool read_task(AuxT& aux, const WaitCtx& w, Ring& r, uint32_t rank, bool warp_wide,
                                          int lane, int4& task)
{
    if (!wait_mbar_cl(w, ptx::smem_u32(&aux.task_full[r.slot]), r.phase, SITE_TASK_FULL))
        return false;
    task = aux.task[r.slot];
    if (warp_wide)
        __syncwarp();
    if (!warp_wide || lane == 0)
        arrive_on_leader(ptx::smem_u32(&aux.task_empty[r.slot]), rank);
    r.advance();
    return true;
}

// Leader's producer: hand a task to this CTA's consumers (a plain store and a
// local arrival) and to the peer CTA's.  The peer's copy travels as one
// asynchronous 16-byte store that completes the peer's slot barrier itself,
// so the producer goes on to its copies without waiting for the remote write.
template <class AuxT>
__device__ __forceinline__ void publish_task(AuxT& aux, Ring& r, int4 task)
{
    aux.task[r.slot] = task;
    ptx::mbar_arrive(ptx::smem_u32(&aux.task_full[r.slot]));
    const uint32_t peer_full = ptx::mapa(ptx::smem_u32(&aux.task_full[r.slot]), 1);
    ptx::mbar_arrive_expect_tx_cluster_relaxed(peer_full, static_cast<uint32_t>(sizeof(int4)));
    ptx::st_async_v4(ptx::mapa(ptx::smem_u32(&aux.task[r.slot]), 1), task, peer_full);
    r.advance();
}

// Layer-2 producer: make sure H chunk j of the band is published, polling a
// window of up to H_WINDOW chunks at once (relaxed loads of this CTA's four
// words per chunk, independent so they overlap), then one acquire fence and
// one proxy fence.  Advances ready_upto past every chunk found ready.
constexpr int H_WINDOW = 8;

static __device__ __noinline__ bool wait_h_chunks(const WaitCtx& w, const uint32_t* band_flags, uint32_t epoch, int j,
                                           int n1, int& ready_upto, uint32_t info)
{
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        const int end = j + H_WINDOW < n1 ? j + H_WINDOW : n1;
        int upto = j;
        bool gap = false;
        for (int c = j; c < end; ++c) {
            const uint32_t* f = band_flags + c * FLAG_WORDS_PER_TILE;
            uint32_t v[EPI_WARPS];
#pragma unroll
            for (int q = 0; q < EPI_WARPS; ++q)
                asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v[q]) : "l"(f + q) : "memory");
            bool all = true;
#pragma unroll
            for (int q = 0; q < EPI_WARPS; ++q)
                all = all && (v[q] == epoch);
            if (!gap && all)
                upto = c + 1;
            else
                gap = true;
        }
        if (upto > j) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            ptx::fence_proxy_async_global();
            ready_upto = upto;
            return true;
        }
        if (*w.abort)
            return false;
        if (ptx::globaltimer() - t0 > w.limit_ns) {
            raise_error(w, static_cast<uint32_t>(TFFN_ERR_TIMEOUT), SITE_H_FLAG, info);
            return false;
        }
        __nanosleep(64);
    }
}

// Whole band of H published for this CTA's rows: one acquire load of the
// band's count instead of a poll over its per-tile flags.
template <int MAX_E>
__device__ __forceinline__ bool band_complete(const Params<MAX_E>& p, int32_t band, uint32_t rank, int32_t n1)
{
    return p.band_count != nullptr &&
           ptx::ld_acquire_gpu(&p.band_count[band * 2 + rank]) == static_cast<uint32_t>(n1 * EPI_WARPS);
}

// ----------------------------------------------------------------- producer
template <int MAX_E>
__device__ void run_producer(const Params<MAX_E>& p, Aux& aux, uint8_t* stages, const WaitCtx& w,
                             int64_t m_blocks, int64_t total, uint32_t rank)
{
    const int32_t n1 = p.layer[0].n_tiles;
    const int32_t n2 = p.layer[1].n_tiles;
    uint32_t stage = 0, phase = 0;
    Ring ring;
    int32_t last_phase[STAGES];
    for (int s = 0; s < STAGES; ++s)
        last_phase[s] = -1;

    // The leader claims tickets one task ahead: when it starts a task, the
    // next one is already claimed and in both CTAs' rings, so the B loader,
    // the MMA thread and the peer move on to it without waiting for the
    // claim.  Holding one ticket ahead keeps the schedule deadlock-free: a
    // pair only holds a ticket larger than the one it runs, and every task
    // waits only on tasks with smaller tickets.
    auto claim_publish = [&](int4& out) -> bool {
        const uint32_t t = atomicAdd(&p.ctrl->ticket, 1u);
        EngineTask et = engine_task_t<int32_t>(static_cast<int32_t>(t), static_cast<int32_t>(m_blocks), n1, n2,
                                               p.group_m, p.mode);
        if (static_cast<int64_t>(t) >= total)
            et.layer = -1;
        out = make_int4(et.layer, et.band, et.tile, 0);
        if (!wait_mbar_cl(w, ptx::smem_u32(&aux.task_empty[ring.slot]), ring.phase ^ 1u, SITE_TASK_EMPTY))
            return false;
        publish_task(aux, ring, out);
        return true;
    };
    int4 ahead = make_int4(-1, 0, 0, 0);
    const bool started = rank != 0 || claim_publish(ahead);
    while (started) {
        int4 task;
        if (rank == 0) {
            task = ahead;
            if (task.x >= 0 && !claim_publish(ahead))
                break;
        } else if (!read_task(aux, w, ring, rank, false, 0, task)) {
            break;
        }
        if (task.x < 0)
            break;

        const int L = task.x;
        const LayerArgs& la = p.layer[L];
        const CUtensorMap* ma = &p.map_a[L];
        const int nk = (la.K + BK - 1) / BK;
        const int32_t row0 = task.y * BM + static_cast<int32_t>(rank) * BM_CTA;
        const bool wait_h = (L == 1 && p.mode == MODE_FUSED);
        // H chunks [0, ready_upto) of this band are known to be published
        int ready_upto = wait_h ? 0 : n1;
        if (wait_h && band_complete(p, task.y, rank, n1)) {
            ptx::fence_proxy_async_global();
            ready_upto = n1;
        }
        const uint32_t* band_flags =
            p.flags + static_cast<uint32_t>(task.y * n1) * FLAG_WORDS_PER_TILE + rank * EPI_WARPS;
        bool ok = true;
        for (int kb = 0; kb < nk && ok; ++kb) {
            // Layer 2 only: the k-block reads H, whose chunk comes from
            // layer-1 tile j (a layer-1 task's k runs over N, not over H).
            const int j = wait_h ? (kb * BK) / h_cols_per_tile(p) : 0;
            if (j >= ready_upto) {
                ok = wait_h_chunks(w, band_flags, aux.epoch, j, n1, ready_upto,
                                   static_cast<uint32_t>(task.y * n1 + j));
                if (!ok)
                    break;
            }
            ok = wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY);
            if (!ok)
                break;
            const uint32_t fb_local = ptx::smem_u32(&aux.full[stage]);
            const uint32_t fb = ptx::mapa(fb_local, 0);     // the leader's stage barrier
            if (rank == 0)
                ptx::mbar_arrive_expect_tx(fb_local, 2 * STAGE_BYTES);
            const uint32_t sa = ptx::smem_u32(stages + stage * STAGE_BYTES);
            ptx::tma_load_2d_pair(sa, ma, fb, kb * BK, row0);
            last_phase[stage] = static_cast<int32_t>(phase);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok)
            break;
    }
    // Exit: every copy of the pair has landed (the leader's stage barriers
    // count both CTAs' bytes; the peer cannot leave before the leader passes
    // the final cluster barrier).
    if (rank == 0)
        for (int s = 0; s < STAGES; ++s)
            if (last_phase[s] >= 0)
                wait_own(w, ptx::smem_u32(&aux.full[s]), static_cast<uint32_t>(last_phase[s]));
}

// ---------------------------------------------------------------- B loader
template <int MAX_E>
__device__ void run_b_loader(const Params<MAX_E>& p, Aux& aux, uint8_t* stages, const WaitCtx& w, uint32_t rank)
{
    uint32_t stage = 0, phase = 0;
    Ring ring;
    for (;;) {
        int4 task;
        if (!read_task(aux, w, ring, rank, false, 0, task))
            break;
        if (task.x < 0)
            break;
        const int L = task.x;
        // A gated layer-1 tile: the leader CTA's B half is W1's 128 columns,
        // the peer's half the same 128 columns of W3.
        const bool gated = p.glu && L == 0;
        const int e = expert_of(p, task.y);
        const CUtensorMap* mb = (gated && rank == 1) ? &p.map_b_lin[e] : &p.map_b[L][e];
        const int nk = (p.layer[L].K + BK - 1) / BK;
        const int32_t col0 = gated ? task.z * BN_CTA : task.z * BN + static_cast<int32_t>(rank) * BN_CTA;
        for (int kb = 0; kb < nk; ++kb) {
            if (!wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY))
                return;
            const uint32_t fb = ptx::mapa(ptx::smem_u32(&aux.full[stage]), 0);   // the leader's barrier
            const uint32_t sb = ptx::smem_u32(stages + stage * STAGE_BYTES) + A_STAGE_BYTES;
            if (p.b3d) {
                ptx::tma_load_3d_pair(sb, mb, fb, 0, kb * BK, col0 / 64);
            } else {
#pragma unroll
                for (int i = 0; i < BN_CTA / 64; ++i)
                    ptx::tma_load_2d_pair(sb + i * B_BOX_BYTES, mb, fb, col0 + i * 64, kb * BK);
            }
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// ------------------------------------------------------------- leader: MMA
template <int MAX_E>
__device__ void run_mma(const Params<MAX_E>& p, Aux& aux, uint8_t* stages, const WaitCtx& w,
                        uint32_t tmem_base)
{
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, 0, 1);
    uint32_t stage = 0, phase = 0, iter = 0;
    Ring ring;
    for (;;) {
        int4 task;
        if (!read_task(aux, w, ring, 0, false, 0, task))
            break;
        if (task.x < 0)
            break;
        const int nk = (p.layer[task.x].K + BK - 1) / BK;
        const uint32_t acc = iter & 1u;
        const uint32_t acc_phase = (iter >> 1) & 1u;
        if (!wait_mbar_cl(w, ptx::smem_u32(&aux.tmem_empty[acc]), acc_phase ^ 1u, SITE_TMEM_EMPTY))
            break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            ok = wait_mbar(w, ptx::smem_u32(&aux.full[stage]), phase, SITE_SMEM_FULL);
            if (!ok)
                break;
            ptx::tc_fence_after();
            const uint32_t sa = ptx::smem_u32(stages + stage * STAGE_BYTES);
            const uint32_t sb = sa + A_STAGE_BYTES;
            // A: K-major, rows of 128 B, 8-row groups 1 KiB apart; a 16-wide
            // k step advances 32 B inside the swizzle atom.
            const uint64_t adesc = ptx::sdesc_sw128(sa, 16, 1024);
            // B: MN-major, 64-column blocks 8 KiB apart (LBO), 8-row k groups
            // 1 KiB apart (SBO); a 16-deep k step advances 2 KiB.
            const uint64_t bdesc = ptx::sdesc_sw128(sb, B_BOX_BYTES, 1024);
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
    // Exit: wait until every MMA this thread issued has completed.
    ptx::umma_commit_pair_mc(ptx::smem_u32(&aux.drain), 0x1);
    wait_own(w, ptx::smem_u32(&aux.drain), 0u);
}

// ----------------------------------------------------------------- epilogue
// The tile's 256 bias values (fp32; zeros outside the matrix and for a NULL
// bias) in one shared slice: epilogue warp q fetches columns [64q, 64q+64),
// two per lane, before the accumulator wait, so the global latency overlaps
// the main loop.
__device__ __forceinline__ void fetch_bias_part(const __nv_bfloat16* bias, int32_t col0, int32_t ncols, float* slice,
                                                uint32_t quad, int lane)
{
    const int32_t i = static_cast<int32_t>(quad) * 64 + lane * 2;
    const int32_t c = col0 + i;
    float2 v = make_float2(0.0f, 0.0f);
    if (bias != nullptr && c < ncols) {   // ncols is even: both columns are inside
        const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(bias + c));
        v = make_float2(bf16_lo(u), bf16_hi(u));
    }
    *reinterpret_cast<float2*>(slice + i) = v;
}

// ---- bf16 outputs through shared memory and TMA stores.
// A staging buffer holds a 32-row x 64-column bf16 box in the 128-byte
// swizzled layout a TMA store reads: 16-byte chunk j (0..7) of row r sits at
// r * 128 + (j ^ (r % 8)) * 16.  Each thread writes its own row, one 32-column
// half (chunks 4h .. 4h+3) at a time.
__device__ __forceinline__ void stage_half(uint32_t buf, int lane, int h, const uint32_t (&pk)[16])
{
    const uint32_t rowaddr = buf + static_cast<uint32_t>(lane) * 128u;
    const uint32_t sw = static_cast<uint32_t>(lane) & 7u;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        ptx::st_shared_v4(rowaddr + (((static_cast<uint32_t>(4 * h + j)) ^ sw) << 4), pk[4 * j], pk[4 * j + 1],
                          pk[4 * j + 2], pk[4 * j + 3]);
}

// Bias, activation and bf16 rounding of 32 accumulator columns into 16 packed
// words (the same arithmetic as store_chunk).
template <int ACT>
__device__ __forceinline__ void convert32(const uint32_t (&acc)[32], uint32_t bias_smem, uint32_t (&pk)[16])
{
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float4 b;   // the same address in every lane: a broadcast
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(b.x), "=f"(b.y), "=f"(b.z), "=f"(b.w)
                     : "r"(bias_smem + q * 16));
        pk[2 * q] = pack_bf16x2(act_apply(ACT, __uint_as_float(acc[q * 4 + 0]) + b.x),
                                act_apply(ACT, __uint_as_float(acc[q * 4 + 1]) + b.y));
        pk[2 * q + 1] = pack_bf16x2(act_apply(ACT, __uint_as_float(acc[q * 4 + 2]) + b.z),
                                    act_apply(ACT, __uint_as_float(acc[q * 4 + 3]) + b.w));
    }
}

// Before a staging buffer is rewritten: the store issued from it two boxes
// ago has finished reading it (lane 0 issued every store of the warp).
__device__ __forceinline__ void out_buffer_free(int lane)
{
    if (lane == 0)
        ptx::bulk_wait_group_read<1>();
    __syncwarp();
}

// The staged box to global memory: every lane's shared-memory writes are made
// visible to the async proxy, then lane 0 issues the store as one bulk group.
// Rows and columns outside the map (past the output's extent) are not written.
__device__ __forceinline__ void out_store_box(const CUtensorMap* map, uint32_t buf, int lane, int32_t x, int32_t y)
{
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        ptx::tma_store_2d(map, buf, x, y);
        ptx::bulk_commit_group();
    }
}

// Drain one accumulator tile through the staging buffers, 64 columns per box;
// the TMEM load of the next 32 columns is in flight while the current ones are
// converted.  Returns the warp's next staging buffer.
template <int ACT>
__device__ __forceinline__ uint32_t drain_tile_tma(uint32_t taddr, int nchunks, uint32_t bias_smem,
                                                   const CUtensorMap* map, uint32_t stage, uint32_t sb, int lane,
                                                   int32_t row0, int32_t col_base)
{
    uint32_t ra[32], rb[32];
    __syncwarp();
    ptx::tmem_ld_32x32b_x32(taddr, ra);
    for (int c = 0; c < nchunks; c += 2) {
        const uint32_t buf = stage + sb * OUT_BUF_BYTES;
        out_buffer_free(lane);
        uint32_t pk[16];
        ptx::tmem_ld_wait();
        if (c + 1 < nchunks)
            ptx::tmem_ld_32x32b_x32(taddr + (c + 1) * 32, rb);
        convert32<ACT>(ra, bias_smem + c * 128, pk);
        stage_half(buf, lane, 0, pk);
        if (c + 1 < nchunks) {
            ptx::tmem_ld_wait();
            if (c + 2 < nchunks)
                ptx::tmem_ld_32x32b_x32(taddr + (c + 2) * 32, ra);
            convert32<ACT>(rb, bias_smem + (c + 1) * 128, pk);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = 0u;   // columns past the output: clipped by the store
        }
        stage_half(buf, lane, 1, pk);
        out_store_box(map, buf, lane, col_base + c * 32, row0);
        sb ^= 1u;
    }
    return sb;
}

// Gated layer-1 tile through the staging buffers: gate columns [0, 128) and
// linear columns [128, 256) of the accumulator give 128 H columns.
template <int ACT>
__device__ __forceinline__ uint32_t drain_glu_tma(uint32_t taddr, int nchunks, const CUtensorMap* map,
                                                  uint32_t stage, uint32_t sb, int lane, int32_t row0,
                                                  int32_t col_base)
{
    for (int c = 0; c < nchunks; c += 2) {
        const uint32_t buf = stage + sb * OUT_BUF_BYTES;
        out_buffer_free(lane);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
            if (c + h < nchunks) {
                uint32_t g[32], u[32];
                __syncwarp();
                ptx::tmem_ld_32x32b_x32(taddr + (c + h) * 32, g);
                ptx::tmem_ld_32x32b_x32(taddr + BN_CTA + (c + h) * 32, u);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(act_apply(ACT, __uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]),
                                        act_apply(ACT, __uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]));
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = 0u;
            }
            stage_half(buf, lane, h, pk);
        }
        out_store_box(map, buf, lane, col_base + c * 32, row0);
        sb ^= 1u;
    }
    return sb;
}

// fp32 output (the MoE experts' Y rows before the weighted sum): a 32-column
// chunk is a full 128-byte row of a 32 x 32 fp32 box, converted in place.
template <int ACT>
__device__ __forceinline__ uint32_t drain_tile_tma_f32(uint32_t taddr, int nchunks, uint32_t bias_smem,
                                                       const CUtensorMap* map, uint32_t stage, uint32_t sb, int lane,
                                                       int32_t row0, int32_t col_base)
{
    const uint32_t sw = static_cast<uint32_t>(lane) & 7u;
    for (int c = 0; c < nchunks; ++c) {
        uint32_t ra[32];
        const uint32_t buf = stage + sb * OUT_BUF_BYTES;
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(taddr + c * 32, ra);
        out_buffer_free(lane);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float4 b;   // the same address in every lane: a broadcast
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(b.x), "=f"(b.y), "=f"(b.z), "=f"(b.w)
                         : "r"(bias_smem + c * 128 + q * 16));
            ptx::st_shared_v4(buf + static_cast<uint32_t>(lane) * 128u + ((static_cast<uint32_t>(q) ^ sw) << 4),
                              __float_as_uint(act_apply(ACT, __uint_as_float(ra[q * 4 + 0]) + b.x)),
                              __float_as_uint(act_apply(ACT, __uint_as_float(ra[q * 4 + 1]) + b.y)),
                              __float_as_uint(act_apply(ACT, __uint_as_float(ra[q * 4 + 2]) + b.z)),
                              __float_as_uint(act_apply(ACT, __uint_as_float(ra[q * 4 + 3]) + b.w)));
        }
        out_store_box(map, buf, lane, col_base + c * 32, row0);
        sb ^= 1u;
    }
    return sb;
}

// A finished accumulator tile through the staging buffers and TMA stores, the
// activation resolved to a template argument once; returns the warp's next
// staging buffer.
__device__ __forceinline__ uint32_t drain_any_tma(int act, bool gated, bool out_f32, uint32_t taddr, int nchunks,
                                                  uint32_t bias_smem, const CUtensorMap* map, uint32_t stage,
                                                  uint32_t sb, int lane, int32_t row0, int32_t col_base)
{
#define TFFN_DRAIN_TMA(A)                                                                              \
    do {                                                                                               \
        if (gated)                                                                                     \
            return drain_glu_tma<A>(taddr, nchunks, map, stage, sb, lane, row0, col_base);       \
        if (out_f32)                                                                                   \
            return drain_tile_tma_f32<A>(taddr, nchunks, bias_smem, map, stage, sb, lane, row0, col_base); \
        return drain_tile_tma<A>(taddr, nchunks, bias_smem, map, stage, sb, lane, row0, col_base); \
    } while (0)
    switch (act) {
    case TFFN_ACT_GELU_TANH: TFFN_DRAIN_TMA(TFFN_ACT_GELU_TANH); break;
    case TFFN_ACT_SILU: TFFN_DRAIN_TMA(TFFN_ACT_SILU); break;
    case TFFN_ACT_RELU: TFFN_DRAIN_TMA(TFFN_ACT_RELU); break;
    default: TFFN_DRAIN_TMA(TFFN_ACT_NONE); break;
    }
#undef TFFN_DRAIN_TMA
    return sb;
}

// Fused MoE combine after a layer-2 tile: each lane's row (routing entry
// t*k+s, or -1 for a padding row) has stored its fp32 outputs of Y column tile
// `tile`; its arrival is counted for (t, tile), and the rows that are the last
// of their token's k rows are then finished by the whole warp, one after
// another: lane l forms columns [8l, 8l+8) of Y[t] = bf16(sum_s w[t,s]
// Yp[pos[t,s]]) in slot order (fp32 fma from 0, the same arithmetic as the
// separate combine kernel, so the result does not depend on which row
// finished last), with coalesced reads of the k expert rows.
template <int MAX_E>
__device__ __noinline__ void combine_rows(const Params<MAX_E>& p, int32_t entry, int32_t tile, int32_t col0,
                                          int32_t ncols, int lane)
{
    const int k = p.comb_k;
    bool last = false;
    if (entry >= 0) {
        uint32_t* cnt = p.comb_cnt + static_cast<int64_t>(entry / k) * p.layer[1].n_tiles + tile;
        __threadfence();   // this row's stores before its arrival
        last = atomicAdd(cnt, 1u) == static_cast<uint32_t>(k - 1);
        if (last)
            *cnt = 0u;     // all k rows have arrived: ready for the next call
    }
    uint32_t m = __ballot_sync(0xffffffffu, last);
    if (m == 0u)
        return;
    __threadfence();       // every other row of those tokens is stored and visible
    const float* yp = static_cast<const float*>(p.layer[1].out);
    const int64_t ld = p.layer[1].ld_out;
    const int32_t col = col0 + lane * 8;
    const bool in = col < ncols;   // ncols is a multiple of 8
    while (m != 0u) {
        const int src = __ffs(m) - 1;
        m &= m - 1u;
        const int64_t t = __shfl_sync(0xffffffffu, entry, src) / k;
        if (!in)
            continue;
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            a[i] = 0.0f;
        for (int sl = 0; sl < k; ++sl) {
            const float g = __ldg(p.comb_w + t * k + sl);
            const float4* v4 =
                reinterpret_cast<const float4*>(yp + static_cast<int64_t>(__ldg(p.comb_pos + t * k + sl)) * ld + col);
            const float4 u = __ldcg(v4), v = __ldcg(v4 + 1);
            a[0] = fmaf(g, u.x, a[0]);
            a[1] = fmaf(g, u.y, a[1]);
            a[2] = fmaf(g, u.z, a[2]);
            a[3] = fmaf(g, u.w, a[3]);
            a[4] = fmaf(g, v.x, a[4]);
            a[5] = fmaf(g, v.y, a[5]);
            a[6] = fmaf(g, v.z, a[6]);
            a[7] = fmaf(g, v.w, a[7]);
        }
        *reinterpret_cast<uint4*>(p.comb_y + t * static_cast<int64_t>(ncols) + col) =
            make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                       pack_bf16x2(a[6], a[7]));
    }
}

template <int MAX_E>
__device__ void run_epilogue(const Params<MAX_E>& p, Aux& aux, const WaitCtx& w, uint32_t tmem_base,
                             uint32_t rank, int warp, int lane, float* bias_slice, uint32_t out_stage)
{
    const uint32_t quad = static_cast<uint32_t>(warp & 3);   // TMEM lanes [32*quad, 32*quad+32)
    const int32_t n1 = p.layer[0].n_tiles;
    uint32_t iter = 0;
    uint32_t sb = 0;   // the warp's next staging buffer
    Ring ring;
    for (;;) {
        int4 task;
        if (!read_task(aux, w, ring, rank, true, lane, task))
            break;
        if (task.x < 0)
            break;
        const int L = task.x;
        const LayerArgs& la = p.layer[L];
        const uint32_t acc = iter & 1u;
        const uint32_t acc_phase = (iter >> 1) & 1u;
        const bool gated = p.glu && L == 0;   // gated layer 1: no bias
        // The shared bias slice: every epilogue warp is done with the previous
        // tile's before any writes this tile's part (bounded waits: a warp
        // that gives up leaves the others to time out, not to hang).
        if (iter > 0 && !wait_mbar(w, ptx::smem_u32(&aux.bias_free), (iter - 1) & 1u, SITE_BIAS))
            break;
        fetch_bias_part(gated ? nullptr : p.bias[L][expert_of(p, task.y)], task.z * BN, la.ncols, bias_slice, quad,
                        lane);
        // Fused MoE combine: this thread's row's routing entry (-1: a padding
        // row, not stored), read before the accumulator wait.
        const bool fuse = MAX_E > 1 && L == 1 && p.comb_cnt != nullptr;
        const int64_t row = static_cast<int64_t>(task.y) * BM + rank * BM_CTA + quad * 32 + lane;
        const int32_t entry = (fuse && row < la.rows) ? __ldg(p.row_entry + row) : -1;
        __syncwarp();
        if (lane == 0)
            ptx::mbar_arrive(ptx::smem_u32(&aux.bias_ready));
        if (!wait_mbar(w, ptx::smem_u32(&aux.tmem_full[acc]), acc_phase, SITE_TMEM_FULL) ||
            !wait_mbar(w, ptx::smem_u32(&aux.bias_ready), iter & 1u, SITE_BIAS))
            break;
        ptx::tc_fence_after();
        // The layer's fields in registers: the TMEM loads below are volatile
        // asm with a memory clobber, which would otherwise force every field
        // to be re-read from the parameter block in every chunk.
        const int32_t ncols = la.ncols;
        const int act = la.act;
        const bool out_f32 = la.out_f32 != 0;
        const int32_t tile_cols = gated ? BN_CTA : BN;
        const int32_t col_base = task.z * tile_cols;
        const int nchunks = ncols - col_base >= tile_cols ? tile_cols / 32 : (ncols - col_base + 31) / 32;
        const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + acc * BN;
        const int32_t row0 = task.y * BM + static_cast<int32_t>(rank) * BM_CTA + static_cast<int32_t>(quad) * 32;
        sb = drain_any_tma(act, gated, out_f32, taddr, nchunks, ptx::smem_u32(bias_slice), &p.map_out[L], out_stage,
                           sb, lane, row0, col_base);
        __syncwarp();
        if (lane == 0)
            ptx::mbar_arrive(ptx::smem_u32(&aux.bias_free));
        // Accumulator drained: hand it back to the leader's MMA thread.
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0)
            arrive_on_leader(ptx::smem_u32(&aux.tmem_empty[acc]), rank);
        ++iter;
        if (fuse) {
            // the warp's rows are in memory (its stores completed, the async
            // proxy's writes ordered before the arrivals) before they are counted
            if (lane == 0) {
                ptx::bulk_wait_group<0>();
                ptx::fence_proxy_async_global();
            }
            __syncwarp();
            combine_rows(p, entry, task.z, col_base, ncols, lane);
        }

        // Layer-1 tile: publish this warp's 32 rows of the H tile by stamping
        // the warp's flag word with the call's epoch (release, gpu scope).
        // The tile's TMA stores (issued by lane 0) complete first.
        if (L == 0 && p.mode == MODE_FUSED) {
            if (lane == 0)
                ptx::bulk_wait_group<0>();
            ptx::fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) {
                const int32_t fi = task.y * n1 + task.z;
                if (fi != p.skip_flag) {
                    __threadfence();
                    ptx::st_release_gpu(&p.flags[fi * FLAG_WORDS_PER_TILE + rank * EPI_WARPS + quad], aux.epoch);
                    // counted after the fence above, which orders the rows
                    // before the count as it does before the flag
                    if (p.band_count != nullptr)
                        ptx::red_relaxed_add_gpu(&p.band_count[task.y * 2 + rank], 1u);
                }
            }
        }
    }
    // Every store of this warp has completed before the CTA can leave, and
    // its band counts are ordered before the CTA's exit count (the last CTA
    // out zeroes them).
    if (lane == 0) {
        ptx::bulk_wait_group<0>();
        __threadfence();
    }
    __syncwarp();
}

// ------------------------------------------------------------------- kernel
template <int MAX_E>
__global__ void __launch_bounds__(NUM_THREADS, 1) engine_kernel(const __grid_constant__ Params<MAX_E> p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Aux& aux = *reinterpret_cast<Aux*>(stages + STAGES * STAGE_BYTES + OUT_BYTES);
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
        for (int s = 0; s < TASK_SLOTS; ++s) {
            ptx::mbar_init(ptx::smem_u32(&aux.task_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.task_empty[s]), TASK_CONSUMERS);
        }
        ptx::mbar_init(ptx::smem_u32(&aux.drain), 1);
        ptx::mbar_init(ptx::smem_u32(&aux.bias_ready), EPI_WARPS);
        ptx::mbar_init(ptx::smem_u32(&aux.bias_free), EPI_WARPS);
        aux.abort = 0u;
        // The epoch lives on the device, so a launch replayed from a CUDA
        // graph still gets a fresh value: every CTA reads it before any CTA
        // can finish (the last CTA out is the only writer).
        aux.epoch = *reinterpret_cast<volatile uint32_t*>(&p.ctrl->epoch) + 1u;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&p.map_a[0]);
        ptx::prefetch_tmap(&p.map_a[1]);
        if (MAX_E == 1) {
            ptx::prefetch_tmap(&p.map_b[0][0]);
            ptx::prefetch_tmap(&p.map_b[1][0]);
            if (p.glu)
                ptx::prefetch_tmap(&p.map_b_lin[0]);
        }
    }
    if (warp == 1) {
        // one collective allocation per CTA pair: both CTAs' warp 1 take part
        ptx::tmem_alloc_pair(ptx::smem_u32(&aux.tmem_base), TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem_base = aux.tmem_base;

    const WaitCtx w{&aux.abort, p.ctrl, p.wait_limit_ns, ptx::mapa(ptx::smem_u32(&aux.abort), rank ^ 1u)};
    const int64_t m_blocks = p.m_blocks >= 0 ? p.m_blocks : static_cast<int64_t>(*p.m_blocks_dev);
    const int64_t total = engine_total_tickets(m_blocks, p.layer[0].n_tiles, p.layer[1].n_tiles, p.mode);

    if (warp == 0) {
        if (lane == 0)
            run_producer(p, aux, stages, w, m_blocks, total, rank);
    } else if (warp == B_LOADER_WARP) {
        if (lane == 0)
            run_b_loader(p, aux, stages, w, rank);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0)
            run_mma(p, aux, stages, w, tmem_base);
    } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
        float* bias_slice = reinterpret_cast<float*>(stages + STAGES * STAGE_BYTES + OUT_BYTES + AUX_BYTES);
        const uint32_t out_stage = ptx::smem_u32(stages + STAGES * STAGE_BYTES) +
                                   static_cast<uint32_t>((warp - 2) * 2 * OUT_BUF_BYTES);
        run_epilogue(p, aux, w, tmem_base, rank, warp, lane, bias_slice, out_stage);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    // The leader's MMAs read the peer's shared memory: neither CTA leaves (or
    // frees its tensor memory) before both are done.
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0) {
        // The last CTA out resets the ticket counter for the next launch.
        __threadfence();
        if (atomicAdd(&p.ctrl->done, 1u) == gridDim.x - 1) {
            p.ctrl->ticket = 0u;
            p.ctrl->done = 0u;
            p.ctrl->epoch = aux.epoch;
            if (p.band_count != nullptr && p.mode == MODE_FUSED) {
                const int64_t mb = p.m_blocks >= 0 ? p.m_blocks : static_cast<int64_t>(*p.m_blocks_dev);
                for (int64_t i = 0; i < 2 * mb; ++i)
                    p.band_count[i] = 0u;
            }
            __threadfence();
        }
    }
}

}  // namespace engine
}  // namespace tffn
