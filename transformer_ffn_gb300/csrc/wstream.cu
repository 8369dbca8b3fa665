// wstream.cu -- the medium-batch weight-streaming kernel on tcgen05 (see
// wstream.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "wstream.cuh"

namespace tffn {
namespace wstream {

struct Aux {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t full1[MAX_STAGES];     // window layer 1: its own ring geometry
    uint64_t empty1[MAX_STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint64_t xfer[EPI_WARPS];       // per epilogue warp: bulk loads of layer-2 parts
    uint32_t tmem_base;
    uint32_t abort;
    uint32_t epoch;     // this launch's ready-flag value (control block's + 1)
};
static_assert(sizeof(Aux) <= 1024, "barrier block");

// This CTA's unit range of a layer: [u0, u1) with slice = u / kch, K chunk =
// u % kch.  A run is the part of the range inside one slice; it accumulates
// in one tensor-memory buffer.
struct Range {
    int64_t u0, u1, kch;
};

__device__ __forceinline__ Range range_of(const Plan& pl, int layer)
{
    const int64_t U = pl.units[layer], G = pl.grid, c = blockIdx.x;
    return Range{range_start(c, U, G), range_start(c + 1, U, G), pl.kch[layer]};
}

__device__ __forceinline__ bool run_first(const Range& r, int64_t u)
{
    return u == r.u0 || u % r.kch == 0;
}

__device__ __forceinline__ bool run_last(const Range& r, int64_t u)
{
    return u + 1 == r.u1 || (u + 1) % r.kch == 0;
}

// Window layer 1: the 64-column hidden blocks [b0, b1) this CTA owns.
struct Blocks {
    int32_t b0, b1;
};

__device__ __forceinline__ Blocks blocks_of(const Plan& pl)
{
    const int64_t c = blockIdx.x, G = pl.grid, n = pl.nblk;
    return Blocks{static_cast<int32_t>(c * n / G), static_cast<int32_t>((c + 1) * n / G)};
}

// Wait, with the whole warp, until every H slice read by the K chunks
// [k0, k0 + count) (cyclic over kch) is ready: all four words equal the
// epoch.  A K chunk of KC rows lies in H slice kc * KC / h_cols.
// With the window layer 1 a K chunk is one 64-column block of H, whose two
// words (its two epilogue warps) must equal the epoch.
__device__ bool wait_h(const WaitCtx& w, const uint32_t* flags, uint32_t epoch, int64_t k0, int64_t count, int64_t kch,
                       int64_t h_slices, int64_t h_cols, bool win, int lane)
{
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        bool mine = true;
        for (int64_t i = lane; i < count && mine; i += 32) {
            const int64_t kc = (k0 + i) % kch;
            const int64_t hs = win ? kc : kc * KC / h_cols;
            if (hs >= h_slices)
                continue;
            const int nw = win ? 2 : EPI_WARPS;
            const uint32_t* f = flags + hs * nw;
            uint32_t v[EPI_WARPS];
#pragma unroll
            for (int q = 0; q < EPI_WARPS; ++q)
                if (q < nw)
                    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v[q]) : "l"(f + q) : "memory");
#pragma unroll
            for (int q = 0; q < EPI_WARPS; ++q)
                mine = mine && (q >= nw || v[q] == epoch);
        }
        if (__all_sync(0xffffffffu, mine))
            break;
        if (__any_sync(0xffffffffu, *w.abort != 0u))
            return false;
        bool late = lane == 0 && ptx::globaltimer() - t0 > w.limit_ns;
        late = __shfl_sync(0xffffffffu, late, 0);
        if (late) {
            if (lane == 0)
                raise_error(w, static_cast<uint32_t>(TFFN_ERR_TIMEOUT), SITE_SLICE_FLAG, static_cast<uint32_t>(k0));
            return false;
        }
        __nanosleep(256);
    }
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    __syncwarp();
    return true;
}

// --------------------------------------------------------------- warp 0: TMA
// Layer 1 streams W1 (and W3) with X; layer 2 first loads the W2 part of its
// first stages (W2 does not depend on H), waits once for every H slice its
// range reads, then streams W2 with H.
template <int NB, bool GLU, bool W2>
__device__ void run_producer(const Params& p, Aux& aux, uint8_t* stages, const WaitCtx& w, int lane)
{
    using Gm = Geo<NB>;
    constexpr int NST = Gm::NST;
    const Plan& pl = p.plan;
    uint32_t stage = 0, phase = 0;
    int32_t last_phase[NST];
    for (int s = 0; s < NST; ++s)
        last_phase[s] = -1;
    uint64_t evict_first = 0;
    if (lane == 0)
        evict_first = ptx::policy_evict_first();
    bool ok = true;

    constexpr uint32_t stage_bytes = static_cast<uint32_t>(Gm::W_BYTES + Gm::X_BYTES);
    // the unit's two 128-column tiles: columns [256s, 256s+256) of W, or for
    // the gated layer 1 columns [128s, 128s+128) of W1 and of W3
    auto issue_w = [&](int layer, int64_t slice, int64_t kc, uint32_t st) {
        const uint32_t fb = ptx::smem_u32(&aux.full[st]);
        const uint32_t sw = ptx::smem_u32(stages + st * Gm::STAGE);
        const int32_t row = static_cast<int32_t>(kc * KC);
        const bool gated = GLU && layer == 0;
        const int32_t col0 = static_cast<int32_t>(slice * (gated ? SLICE : 2 * SLICE));
        const CUtensorMap* m0 = &p.map_w[layer];
        const CUtensorMap* m1 = gated ? &p.map_w3 : &p.map_w[layer];
        const int32_t col1 = gated ? col0 : col0 + SLICE;
        ptx::tma_load_2d_hint(sw, m0, fb, col0, row, evict_first);
        ptx::tma_load_2d_hint(sw + W_BOX, m0, fb, col0 + 64, row, evict_first);
        ptx::tma_load_2d_hint(sw + 2 * W_BOX, m1, fb, col1, row, evict_first);
        ptx::tma_load_2d_hint(sw + 3 * W_BOX, m1, fb, col1 + 64, row, evict_first);
    };
    auto issue_x = [&](int layer, int64_t kc, uint32_t st) {
        const uint32_t fb = ptx::smem_u32(&aux.full[st]);
        const uint32_t sx = ptx::smem_u32(stages + st * Gm::STAGE) + Gm::W_BYTES;
        ptx::tma_load_2d(sx, &p.map_x[layer], fb, static_cast<int32_t>(kc * KC), 0);
    };
    auto advance = [&]() {
        if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
        }
    };

    // ---- layer 1
    if (lane == 0 && pl.win) {
        // The window: every K chunk of this CTA's window (W1's 128 columns,
        // and W3's same 128 when gated, or W1's 256 for a four-block window)
        // with the X chunk, in the layer-1 ring.
        constexpr bool two = GLU || W2;   // two 128-column tiles per stage
        constexpr int N1 = two ? Gm::NST : Gm::NST1;
        constexpr int S1 = two ? Gm::STAGE : Gm::STAGE1;
        constexpr uint32_t bytes1 = static_cast<uint32_t>((two ? 4 : 2) * W_BOX + Gm::X_BYTES);
        const Blocks bk = blocks_of(pl);
        uint32_t st1 = 0, ph1 = 0;
        int32_t last1[N1];
        for (int s = 0; s < N1; ++s)
            last1[s] = -1;
        if (bk.b1 > bk.b0) {
            const int32_t col0 = bk.b0 * 64;
            // every CTA walks K in the same order: all windows read the same
            // rows of W1 at about the same time (a CTA-staggered order,
            // tried, was 13 % slower)
            for (int64_t i = 0; i < pl.kch[0]; ++i) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.empty1[st1]), ph1 ^ 1u, SITE_SMEM_EMPTY);
                if (!ok)
                    break;
                const uint32_t fb = ptx::smem_u32(&aux.full1[st1]);
                const uint32_t sw = ptx::smem_u32(stages + st1 * S1);
                const int32_t row = static_cast<int32_t>(i * KC);
                ptx::mbar_arrive_expect_tx(fb, bytes1);
                ptx::tma_load_2d_hint(sw, &p.map_w[0], fb, col0, row, evict_first);
                ptx::tma_load_2d_hint(sw + W_BOX, &p.map_w[0], fb, col0 + 64, row, evict_first);
                if (two) {
                    const CUtensorMap* m1 = GLU ? &p.map_w3 : &p.map_w[0];
                    const int32_t col1 = GLU ? col0 : col0 + 128;
                    ptx::tma_load_2d_hint(sw + 2 * W_BOX, m1, fb, col1, row, evict_first);
                    ptx::tma_load_2d_hint(sw + 3 * W_BOX, m1, fb, col1 + 64, row, evict_first);
                }
                ptx::tma_load_2d(sw + (two ? 4 : 2) * W_BOX, &p.map_x[0], fb, row, 0);
                last1[st1] = static_cast<int32_t>(ph1);
                if (++st1 == N1) {
                    st1 = 0;
                    ph1 ^= 1u;
                }
            }
        }
        // Layer 2's ring reuses this memory: every layer-1 stage consumed
        // first (or, after a failure, at least landed).
        for (int s = 0; s < N1; ++s) {
            if (last1[s] < 0)
                continue;
            if (ok) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.empty1[s]), static_cast<uint32_t>(last1[s]), SITE_SMEM_EMPTY);
            }
            if (!ok) {
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(ptx::smem_u32(&aux.full1[s]), static_cast<uint32_t>(last1[s])))
                    if (ptx::globaltimer() - t0 > p.wait_limit_ns)
                        break;
            }
        }
    } else if (lane == 0) {
        const Range r = range_of(pl, 0);
        for (int64_t u = r.u0; u < r.u1; ++u) {
            ok = wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY);
            if (!ok)
                break;
            ptx::mbar_arrive_expect_tx(ptx::smem_u32(&aux.full[stage]), stage_bytes);
            issue_w(0, u / r.kch, u % r.kch, stage);
            issue_x(0, u % r.kch, stage);
            last_phase[stage] = static_cast<int32_t>(phase);
            advance();
        }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;

    // ---- layer 2
    if (ok) {
        const Range r = range_of(pl, 1);
        const int64_t npre = (r.u1 - r.u0) < NST ? (r.u1 - r.u0) : NST;
        uint32_t pre_stage[NST];
        if (lane == 0) {
            for (int64_t i = 0; i < npre; ++i) {
                const int64_t u = r.u0 + i;
                ok = wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY);
                if (!ok)
                    break;
                ptx::mbar_arrive_expect_tx(ptx::smem_u32(&aux.full[stage]), stage_bytes);
                issue_w(1, u / r.kch, u % r.kch, stage);
                pre_stage[i] = stage;
                last_phase[stage] = static_cast<int32_t>(phase);
                advance();
            }
        }
        const int npre_done = __shfl_sync(0xffffffffu, ok ? static_cast<int>(npre) : -1, 0);
        if (npre_done >= 0) {
            const int64_t count = (r.u1 - r.u0) < r.kch ? (r.u1 - r.u0) : r.kch;
            const bool ready =
                wait_h(w, p.flags, aux.epoch, r.u0 % r.kch, count, r.kch, pl.win ? pl.nblk : pl.slices[0], pl.h_cols,
                       pl.win != 0, lane);
            if (lane == 0) {
                ptx::fence_proxy_async_global();
                // the prefetched stages expect their H bytes: issue them even
                // after a failed wait so that every barrier completes
                for (int64_t i = 0; i < npre; ++i)
                    issue_x(1, (r.u0 + i) % r.kch, pre_stage[i]);
                if (ready) {
                    for (int64_t u = r.u0 + npre; u < r.u1; ++u) {
                        if (!wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY))
                            break;
                        ptx::mbar_arrive_expect_tx(ptx::smem_u32(&aux.full[stage]), stage_bytes);
                        issue_w(1, u / r.kch, u % r.kch, stage);
                        issue_x(1, u % r.kch, stage);
                        last_phase[stage] = static_cast<int32_t>(phase);
                        advance();
                    }
                }
            }
        }
    }

    // Exit: every copy issued by this warp has landed before the CTA leaves.
    if (lane == 0) {
        for (int s = 0; s < NST; ++s) {
            if (last_phase[s] < 0)
                continue;
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(ptx::smem_u32(&aux.full[s]), static_cast<uint32_t>(last_phase[s]))) {
                if (ptx::globaltimer() - t0 > p.wait_limit_ns) {
                    raise_error(w, static_cast<uint32_t>(TFFN_ERR_TIMEOUT), SITE_DRAIN, s);
                    break;
                }
            }
        }
    }
}

// -------------------------------------------------------- warp 1: the MMAs
// Per unit and tile: four k steps of D[128 x NB] += W^T[128 x 16] X^T[16 x NB];
// A is the MN-major W tile (two 64-column blocks, W_BOX apart; 8-row k groups
// 1 KiB apart; a 16-deep k step advances 2 KiB), B the K-major X tile (rows
// of 128 bytes; a k step advances 32 bytes), shared by both tiles, whose
// products go to the two NB-column halves of the run's buffer.
template <int NB, bool GLU, bool W2>
__device__ void run_mma(const Params& p, Aux& aux, uint8_t* stages, const WaitCtx& w, uint32_t tmem_base)
{
    using Gm = Geo<NB>;
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(SLICE, NB, 1, 0);
    const Plan& pl = p.plan;
    uint32_t stage = 0, phase = 0, iter = 0;
    bool ok = true;
    for (int layer = 0; layer < 2 && ok; ++layer) {
        if (layer == 0 && pl.win) {
            // the window: one run over all K chunks, in the layer-1 ring
            constexpr bool two = GLU || W2;
            constexpr int N1 = two ? Gm::NST : Gm::NST1;
            constexpr int S1 = two ? Gm::STAGE : Gm::STAGE1;
            const Blocks bk = blocks_of(pl);
            if (bk.b1 <= bk.b0)
                continue;
            const uint32_t buf = iter % Gm::NBUF;
            ok = wait_mbar(w, ptx::smem_u32(&aux.tmem_empty[buf]), ((iter / Gm::NBUF) & 1u) ^ 1u, SITE_TMEM_EMPTY);
            if (!ok)
                break;
            ptx::tc_fence_after();
            const uint32_t d = tmem_base + buf * Gm::ACC_COLS;
            uint32_t st1 = 0, ph1 = 0;
            for (int64_t kc = 0; kc < pl.kch[0]; ++kc) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.full1[st1]), ph1, SITE_SMEM_FULL);
                if (!ok)
                    break;
                ptx::tc_fence_after();
                const uint32_t sw = ptx::smem_u32(stages + st1 * S1);
                const uint64_t adesc = ptx::sdesc_sw128(sw, W_BOX, 1024);
                const uint64_t adesc1 = ptx::sdesc_sw128(sw + 2 * W_BOX, W_BOX, 1024);
                const uint64_t bdesc = ptx::sdesc_sw128(sw + (two ? 4 : 2) * W_BOX, 16, 1024);
#pragma unroll
                for (int k = 0; k < KC / 16; ++k) {
                    const uint64_t bk16 = bdesc + static_cast<uint64_t>((k * 32) >> 4);
                    const uint32_t acc = (kc == 0 && k == 0) ? 0u : 1u;
                    ptx::umma_bf16(d, adesc + static_cast<uint64_t>((k * 2048) >> 4), bk16, idesc, acc);
                    if (two)
                        ptx::umma_bf16(d + NB, adesc1 + static_cast<uint64_t>((k * 2048) >> 4), bk16, idesc, acc);
                }
                ptx::umma_commit(ptx::smem_u32(&aux.empty1[st1]));
                if (++st1 == N1) {
                    st1 = 0;
                    ph1 ^= 1u;
                }
            }
            if (ok)
                ptx::umma_commit(ptx::smem_u32(&aux.tmem_full[buf]));
            ++iter;
            continue;
        }
        const Range r = range_of(pl, layer);
        for (int64_t u = r.u0; u < r.u1; ++u) {
            const bool first = run_first(r, u);
            const uint32_t buf = iter % Gm::NBUF;
            if (first) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.tmem_empty[buf]), ((iter / Gm::NBUF) & 1u) ^ 1u, SITE_TMEM_EMPTY);
                if (!ok)
                    break;
                ptx::tc_fence_after();
            }
            ok = wait_mbar(w, ptx::smem_u32(&aux.full[stage]), phase, SITE_SMEM_FULL);
            if (!ok)
                break;
            ptx::tc_fence_after();
            const uint32_t sw = ptx::smem_u32(stages + stage * Gm::STAGE);
            const uint32_t sx = sw + Gm::W_BYTES;
            const uint32_t d = tmem_base + buf * Gm::ACC_COLS;
            const uint64_t adesc = ptx::sdesc_sw128(sw, W_BOX, 1024);
            const uint64_t bdesc = ptx::sdesc_sw128(sx, 16, 1024);
            const uint64_t adesc1 = ptx::sdesc_sw128(sw + 2 * W_BOX, W_BOX, 1024);
#pragma unroll
            for (int k = 0; k < KC / 16; ++k) {
                const uint64_t bk = bdesc + static_cast<uint64_t>((k * 32) >> 4);
                const uint32_t acc = (first && k == 0) ? 0u : 1u;
                ptx::umma_bf16(d, adesc + static_cast<uint64_t>((k * 2048) >> 4), bk, idesc, acc);
                ptx::umma_bf16(d + NB, adesc1 + static_cast<uint64_t>((k * 2048) >> 4), bk, idesc, acc);
            }
            ptx::umma_commit(ptx::smem_u32(&aux.empty[stage]));
            if (++stage == Gm::NST) {
                stage = 0;
                phase ^= 1u;
            }
            if (run_last(r, u)) {
                ptx::umma_commit(ptx::smem_u32(&aux.tmem_full[buf]));
                ++iter;
            }
        }
    }
    // Exit: wait until every MMA this thread issued has completed.
    ptx::umma_commit(ptx::smem_u32(&aux.drain));
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(ptx::smem_u32(&aux.drain), 0u)) {
        if (ptx::globaltimer() - t0 > p.wait_limit_ns) {
            raise_error(w, static_cast<uint32_t>(TFFN_ERR_TIMEOUT), SITE_DRAIN, 0xFFu);
            break;
        }
    }
}

// -------------------------------------------------------- warps 2-5: drain
// The epilogue works on chunks of CH token rows of this thread's column.
constexpr int CH = 16;

// Output values of CH tokens for this thread's column: act(v + bias), or
// act(gate) * linear for the gated layer 1, rounded to bf16.  Two lanes (two
// adjacent columns) swap halves of their row pairs so that each stores one
// 4-byte column pair of one row.  The activation is a template argument,
// resolved once per run.
constexpr int ACT_RUNTIME = -1;   // the activation read at run time (rarely used gated forms)

template <int ACT, bool GATED>
__device__ __forceinline__ void store_chunk(__nv_bfloat16* out, int ncols, int M, int64_t gcol, float bias,
                                            float (&v)[CH], const float (&lin)[CH], int t0, int lane, int act_rt)
{
    const bool col_ok = gcol < ncols;   // ncols is a multiple of 8: a pair is in or out together
    const int act = ACT == ACT_RUNTIME ? act_rt : ACT;
#pragma unroll
    for (int i = 0; i < CH; ++i)
        v[i] = GATED ? act_apply(act, v[i]) * lin[i] : act_apply(act, v[i] + bias);
#pragma unroll
    for (int i = 0; i < CH; i += 2) {
        const __nv_bfloat162 mine = __floats2bfloat162_rn(v[i], v[i + 1]);   // rows i, i+1 of my column
        const uint32_t m = *reinterpret_cast<const uint32_t*>(&mine);
        const uint32_t o = __shfl_xor_sync(0xffffffffu, m, 1);              // the partner column's pair
        // even lane: row i of (my column, partner column); odd lane: row i+1
        const uint32_t w = (lane & 1) == 0 ? ((m & 0xFFFFu) | (o << 16)) : ((o >> 16) | (m & 0xFFFF0000u));
        const int t = t0 + i + (lane & 1);
        if (col_ok && t < M)
            *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(t) * ncols + (gcol & ~static_cast<int64_t>(1))) = w;
    }
}

__device__ __forceinline__ void tmem_chunk(uint32_t taddr, float (&v)[CH])
{
    uint32_t r[CH];
    ptx::tmem_ld_32x32b_x16(taddr, r);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < CH; ++i)
        v[i] = __uint_as_float(r[i]);
}

// store_chunk with the activation chosen at run time, once per chunk: the
// dense activations and SwiGLU's SiLU compiled in, the rarer gated forms
// (GeGLU, ReGLU, bilinear) through the run-time activation.
template <bool GATED>
__device__ __forceinline__ void store_any(int act, __nv_bfloat16* out, int ncols, int M, int64_t gcol, float bias,
                                          float (&v)[CH], const float (&lin)[CH], int t0, int lane)
{
    if constexpr (GATED) {
        if (act == TFFN_ACT_SILU)
            store_chunk<TFFN_ACT_SILU, true>(out, ncols, M, gcol, bias, v, lin, t0, lane, act);
        else
            store_chunk<ACT_RUNTIME, true>(out, ncols, M, gcol, bias, v, lin, t0, lane, act);
    } else {
        switch (act) {
        case TFFN_ACT_RELU: store_chunk<TFFN_ACT_RELU, false>(out, ncols, M, gcol, bias, v, lin, t0, lane, act); break;
        case TFFN_ACT_GELU_TANH:
            store_chunk<TFFN_ACT_GELU_TANH, false>(out, ncols, M, gcol, bias, v, lin, t0, lane, act);
            break;
        case TFFN_ACT_SILU: store_chunk<TFFN_ACT_SILU, false>(out, ncols, M, gcol, bias, v, lin, t0, lane, act); break;
        default: store_chunk<TFFN_ACT_NONE, false>(out, ncols, M, gcol, bias, v, lin, t0, lane, act); break;
        }
    }
}

// acc[4i .. 4i+3] = sum over parts pp = 0 .. nparts-1, in that order, of the
// float4 at src + pp * pf + i * 32 * 4 (src: this lane's float4 of its
// segment); F parts' loads in flight.
template <int F>
__device__ __forceinline__ void sum_parts(float (&acc)[CH], const float* src, int64_t pf, int nparts)
{
#pragma unroll
    for (int i = 0; i < CH; ++i)
        acc[i] = 0.0f;
#pragma unroll 1
    for (int pp = 0; pp < nparts; pp += F) {
        float4 x[F][CH / 4];
#pragma unroll
        for (int j = 0; j < F; ++j)
            if (pp + j < nparts) {
                const float4* sj = reinterpret_cast<const float4*>(src + static_cast<int64_t>(pp + j) * pf);
#pragma unroll
                for (int i = 0; i < CH / 4; ++i)
                    x[j][i] = __ldcg(sj + i * 32);
            }
#pragma unroll
        for (int j = 0; j < F; ++j)
            if (pp + j < nparts) {
#pragma unroll
                for (int i = 0; i < CH / 4; ++i) {
                    acc[4 * i] += x[j][i].x;
                    acc[4 * i + 1] += x[j][i].y;
                    acc[4 * i + 2] += x[j][i].z;
                    acc[4 * i + 3] += x[j][i].w;
                }
            }
    }
}

// Where a run of this CTA stands in its slice.
struct RunInfo {
    int nparts, part;
};

__device__ __forceinline__ RunInfo run_info(const Plan& pl, int layer, int64_t slice)
{
    const int64_t U = pl.units[layer], G = pl.grid, kch = pl.kch[layer];
    const int64_t first = owner_of(slice * kch, U, G);
    const int64_t last = owner_of((slice + 1) * kch - 1, U, G);
    return RunInfo{static_cast<int>(last - first + 1), static_cast<int>(blockIdx.x - first)};
}

// Per slice and epilogue warp: an arrival counter (parts stored) and a done
// counter (shares summed); both back to zero when the slice is finished.
__device__ __forceinline__ uint32_t* arrive_counter(const Params& p, int layer, int64_t slice, int q)
{
    return p.counters + (layer == 0 ? 0 : p.plan.slices[0] * EPI_WARPS) + slice * EPI_WARPS + q;
}

__device__ __forceinline__ uint32_t* done_counter(const Params& p, int layer, int64_t slice, int q)
{
    return arrive_counter(p, layer, slice, q) + (p.plan.slices[0] + p.plan.slices[1]) * EPI_WARPS;
}

// The output columns of this thread in a slice (two halves, or one gated
// column) and their biases.
struct Cols {
    int64_t gcol[2];
    float bias[2];
};

template <bool GATED>
__device__ __forceinline__ Cols cols_of(const Params& p, int layer, int64_t slice, int col)
{
    Cols c;
    const int ncols = layer == 0 ? p.O : p.P;
    const __nv_bfloat16* b = GATED ? nullptr : (layer == 0 ? p.b1 : p.b2);
    for (int a = 0; a < 2; ++a) {
        c.gcol[a] = GATED ? slice * SLICE + col : slice * 2 * SLICE + a * SLICE + col;
        c.bias[a] = (b != nullptr && c.gcol[a] < ncols) ? __bfloat162float(b[c.gcol[a]]) : 0.0f;
    }
    return c;
}

// Layer 1: publish this warp's columns of an H slice (read by TMA in layer 2).
__device__ __forceinline__ void publish_h(const Params& p, const Aux& aux, int64_t slice, int q, int lane)
{
    ptx::fence_proxy_async_global();
    __syncwarp();   // the warp's stores, then one release by lane 0
    if (lane == 0)
        ptx::st_release_gpu(p.flags + slice * EPI_WARPS + q, aux.epoch);
}

// Phase 1 of a run (this thread: column col of each 128-column half, NB token
// rows): when one CTA owns the slice, straight to bf16 output; else this
// part's partial sums go to their fixed place and the slice's arrival counter
// counts them.  Gated: the two halves are the gate and the linear product of
// the same column.
template <int NB, bool GATED>
__device__ void drain_run(const Params& p, Aux& aux, uint32_t tmem_base, int layer, int64_t slice, uint32_t buf, int q,
                          int lane)
{
    using Gm = Geo<NB>;
    const Plan& pl = p.plan;
    const int col = q * 32 + lane;
    const RunInfo ri = run_info(pl, layer, slice);
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Gm::ACC_COLS;
    float v[CH], lin[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i)
        lin[i] = 0.0f;
    if (ri.nparts == 1) {
        const Cols c = cols_of<GATED>(p, layer, slice, col);
        const int ncols = layer == 0 ? p.O : p.P;
        __nv_bfloat16* out = layer == 0 ? p.H : p.Y;
#pragma unroll 1
        for (int a = 0; a < (GATED ? 1 : 2); ++a)
#pragma unroll 1
            for (int ch = 0; ch < NB / CH; ++ch) {
                tmem_chunk(tb + a * NB + ch * CH, v);
                if (GATED)
                    tmem_chunk(tb + NB + ch * CH, lin);
                store_any<GATED>(layer == 0 ? p.act1 : p.act2, out, ncols, p.M, c.gcol[a], c.bias[a], v, lin,
                                 ch * CH, lane);
            }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0)
            ptx::mbar_arrive(ptx::smem_u32(&aux.tmem_empty[buf]));
        if (layer == 0)
            publish_h(p, aux, slice, q, lane);
        return;
    }
    float* mine = p.partial + pl.part_off[layer] + (slice * pl.maxp[layer] + ri.part) * part_floats(NB);
#pragma unroll 1
    for (int a = 0; a < 2; ++a)
#pragma unroll 1
        for (int ch = 0; ch < NB / CH; ++ch) {
            tmem_chunk(tb + a * NB + ch * CH, v);
            float4* dst = reinterpret_cast<float4*>(mine + seg_off<NB>(q, a, ch)) + lane;
#pragma unroll
            for (int i = 0; i < CH / 4; ++i)
                dst[i * 32] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        ptx::mbar_arrive(ptx::smem_u32(&aux.tmem_empty[buf]));
        // the warp's partial sums are published by this one release (the
        // __syncwarp above orders them before it)
        ptx::red_release_add_gpu(arrive_counter(p, layer, slice, q), 1u);
    }
}

// Phase 2 of a split run: once every part of the slice has arrived, this CTA
// sums its share of the slice's chunks (chunk items part, part + nparts, ...)
// over all parts in part order and writes them.  The CTA whose share finishes
// last resets the slice's counters and, in layer 1, publishes the H slice.
// Wait for a warp's bulk loads after a failed wait (abort elsewhere): the
// copies still land in this CTA's shared memory, so it may not leave first.
__device__ void settle_xfer(const Params& p, uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer() - t0 > p.wait_limit_ns)
            break;
}

template <int NB, bool GATED, bool PIPE>
__device__ bool reduce_share(const Params& p, Aux& aux, const WaitCtx& w, uint8_t* ring, uint32_t& xphase, int layer,
                             int64_t slice, int q, int lane)
{
    const Plan& pl = p.plan;
    const int col = q * 32 + lane;
    const RunInfo ri = run_info(pl, layer, slice);
    if (ri.nparts == 1)
        return true;
    uint32_t* arrive = arrive_counter(p, layer, slice, q);
    const Cols c = cols_of<GATED>(p, layer, slice, col);   // the bias loads overlap the wait
    bool ok = true;
    if (lane == 0)
        ok = wait_flag(w, arrive, static_cast<uint32_t>(ri.nparts), SITE_PARTS, static_cast<uint32_t>(slice));
    if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0)
        return false;
    __syncwarp();   // lane 0's acquire covers the warp's reads of the parts
    const int ncols = layer == 0 ? p.O : p.P;
    __nv_bfloat16* out = layer == 0 ? p.H : p.Y;
    const int64_t pf = part_floats(NB);
    const float* base = p.partial + pl.part_off[layer] + slice * pl.maxp[layer] * pf;
    constexpr int NCH = NB / CH;
    const int items = (GATED ? 1 : 2) * NCH;
    float v[CH], lin[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i)
        lin[i] = 0.0f;
    // This part's block of the slice's items: a CTA with two split slices in
    // this layer has two shares to sum, so its blocks are half as long.
    int64_t wsum = 0, wmine = 0;
    const int64_t first_cta = static_cast<int64_t>(blockIdx.x) - ri.part;
    for (int j = 0; j < ri.nparts; ++j) {
        const int64_t wj = pl.split[layer][first_cta + j] > 1 ? 1 : 2;
        if (j < ri.part)
            wmine += wj;
        wsum += wj;
    }
    const int it0 = static_cast<int>(items * wmine / wsum);
    const int it1 = static_cast<int>(items * (wmine + (pl.split[layer][blockIdx.x] > 1 ? 1 : 2)) / wsum);
    const int act = layer == 0 ? p.act1 : p.act2;
    if (!GATED && !PIPE && layer == 1) {
        // Layer 2 ends the kernel: the ring is idle, and each warp fetches its
        // segments of the parts with bulk copies into its quarter of it, as
        // many items (all their parts) at a time as fit, then sums from there.
        // (Used by the gated instance, whose registers leave no room for the
        // two-deep register pipeline below; for the dense instance that
        // pipeline measured faster.)
        constexpr int NCHK = NB / CH;
        const int nparts = ri.nparts;
        uint8_t* reg = ring + q * Geo<NB>::WREG;
        const uint32_t bar = ptx::smem_u32(&aux.xfer[q]);
        const int pcap = Geo<NB>::WSEGS;
        const int ipb = nparts <= pcap ? pcap / nparts : 1;
        if (lane == 0)
            ptx::fence_proxy_async_global();   // the acquired parts, before the copies read them
#pragma unroll 1
        for (int ib = it0; ib < it1; ib += ipb) {
            const int n = (it1 - ib) < ipb ? (it1 - ib) : ipb;
#pragma unroll 1
            for (int p0 = 0; p0 < nparts; p0 += pcap) {   // several rounds only when one item's parts do not fit
                const int p1 = (nparts - p0) < pcap ? nparts : p0 + pcap;
                const int np = p1 - p0;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * np) * 2048u);
                    for (int j = 0; j < n; ++j)
                        for (int pp = p0; pp < p1; ++pp)
                            ptx::bulk_load(ptx::smem_u32(reg + (j * np + (pp - p0)) * 2048),
                                           base + static_cast<int64_t>(pp) * pf +
                                               seg_off<NB>(q, (ib + j) / NCHK, (ib + j) % NCHK),
                                           2048u, bar);
                }
                if (!wait_mbar(w, bar, xphase, SITE_PARTS)) {
                    if (lane == 0)
                        settle_xfer(p, bar, xphase);
                    __syncwarp();
                    return false;
                }
                xphase ^= 1u;
#pragma unroll 1
                for (int j = 0; j < n; ++j) {
                    const int it = ib + j;
                    if (p0 == 0) {
#pragma unroll
                        for (int i = 0; i < CH; ++i)
                            v[i] = 0.0f;
                    }
#pragma unroll 1
                    for (int pp = 0; pp < np; ++pp) {
                        const float4* sv = reinterpret_cast<const float4*>(reg + (j * np + pp) * 2048) + lane;
#pragma unroll
                        for (int i = 0; i < CH / 4; ++i) {
                            const float4 x = sv[i * 32];
                            v[4 * i] += x.x;
                            v[4 * i + 1] += x.y;
                            v[4 * i + 2] += x.z;
                            v[4 * i + 3] += x.w;
                        }
                    }
                    if (p1 == nparts)
                        store_any<false>(act, out, ncols, p.M, c.gcol[it / NCHK], c.bias[it / NCHK], v, lin,
                                         (it % NCHK) * CH, lane);
                }
                __syncwarp();   // every lane has read the region before lane 0 refills it
            }
        }
    } else if constexpr (GATED || !PIPE) {
        // the gated instance (gate and linear sums, both kernels' layers) keeps
        // the plain loop: the registers
#pragma unroll 1
        for (int it = it0; it < it1; ++it) {
            const int a = GATED ? 0 : it / NCH, ch = it % NCH;
            sum_parts<2>(v, base + seg_off<NB>(q, a, ch) + lane * 4, pf, ri.nparts);
            if (GATED)
                sum_parts<2>(lin, base + seg_off<NB>(q, 1, ch) + lane * 4, pf, ri.nparts);
            store_any<GATED>(act, out, ncols, p.M, c.gcol[a], c.bias[a], v, lin, ch * CH, lane);
        }
    } else {
        // Items in a two-deep pipeline: the first four parts of item it + 1
        // are loading while item it is summed and stored.
        float4 xa[4][CH / 4], xb[4][CH / 4];
        auto load4 = [&](float4 (&x)[4][CH / 4], int it, int pp0) {
            const float* src = base + seg_off<NB>(q, it / NCH, it % NCH) + lane * 4;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (pp0 + j < ri.nparts) {
                    const float4* sj = reinterpret_cast<const float4*>(src + static_cast<int64_t>(pp0 + j) * pf);
#pragma unroll
                    for (int i = 0; i < CH / 4; ++i)
                        x[j][i] = __ldcg(sj + i * 32);
                }
        };
        auto add4 = [&](const float4 (&x)[4][CH / 4], int pp0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (pp0 + j < ri.nparts) {
#pragma unroll
                    for (int i = 0; i < CH / 4; ++i) {
                        v[4 * i] += x[j][i].x;
                        v[4 * i + 1] += x[j][i].y;
                        v[4 * i + 2] += x[j][i].z;
                        v[4 * i + 3] += x[j][i].w;
                    }
                }
        };
        auto item = [&](float4 (&cur)[4][CH / 4], float4 (&nxt)[4][CH / 4], int it) {
            if (it + 1 < it1)
                load4(nxt, it + 1, 0);
#pragma unroll
            for (int i = 0; i < CH; ++i)
                v[i] = 0.0f;
            add4(cur, 0);
            for (int pp = 4; pp < ri.nparts; pp += 4) {   // parts past the first four (part order kept)
                load4(cur, it, pp);
                add4(cur, pp);
            }
            const int a = it / NCH;
            store_any<false>(act, out, ncols, p.M, c.gcol[a], c.bias[a], v, lin, (it % NCH) * CH, lane);
        };
        if (it0 < it1)
            load4(xa, it0, 0);
#pragma unroll 1
        for (int it = it0; it < it1; it += 2) {
            item(xa, xb, it);
            if (it + 1 < it1)
                item(xb, xa, it + 1);
        }
    }
    if (layer == 0)
        ptx::fence_proxy_async_global();
    __syncwarp();
    if (lane == 0) {
        uint32_t* done = done_counter(p, layer, slice, q);
        // acquire-release: the last share also sees every other share's stores
        if (ptx::atom_add_acq_rel_gpu(done, 1u) == static_cast<uint32_t>(ri.nparts - 1)) {
            // every share is written (and every CTA is past its wait)
            *arrive = 0u;
            *done = 0u;
            if (layer == 0)
                ptx::st_release_gpu(p.flags + slice * EPI_WARPS + q, aux.epoch);
        }
    }
    __syncwarp();
    return true;
}

// The activation of a run, resolved once; the gated FFN's layer 2 has no bias
// and no activation (ffn_glu_forward), so the gated instance only needs the
// gated layer-1 variants and that one.
// The gated FFN's layer 1 is the gated variant; its layer 2 (no bias, no
// activation) and every dense layer the plain one.
template <int NB, bool GLU, int PHASE>
__device__ __forceinline__ bool run_phase(const Params& p, Aux& aux, const WaitCtx& w, uint8_t* ring, uint32_t& xphase,
                                          uint32_t tmem_base, int layer, int64_t slice, uint32_t buf, int q, int lane)
{
    if (GLU && layer == 0) {
        if (PHASE == 1)
            drain_run<NB, GLU>(p, aux, tmem_base, layer, slice, buf, q, lane);
        else
            return reduce_share<NB, GLU, false>(p, aux, w, ring, xphase, layer, slice, q, lane);
        return true;
    }
    if (PHASE == 1)
        drain_run<NB, false>(p, aux, tmem_base, layer, slice, buf, q, lane);
    else
        return reduce_share<NB, false, !GLU>(p, aux, w, ring, xphase, layer, slice, q, lane);
    return true;
}

// Window layer 1: the CTA's window of H over all of K, one 128-column tile
// (or, for a four-block window, two: tensor-memory columns [0, NB) and
// [NB, 2 NB)).  Warp q holds columns 32q .. 32q + 31 of each tile, in block
// (the tile's first block) + q / 2; the warps of an owned block write it
// (act(v + bias), or act(gate) * linear) and publish its ready word, the
// others only release the accumulator.
template <int NB, bool GATED, bool W2>
__device__ void drain_window(const Params& p, Aux& aux, uint32_t tmem_base, Blocks bk, uint32_t buf, int q, int lane)
{
    using Gm = Geo<NB>;
    constexpr int ntile = (!GATED && W2) ? 2 : 1;
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Gm::ACC_COLS;
#pragma unroll 1
    for (int t = 0; t < ntile; ++t) {
        const int32_t block = bk.b0 + 2 * t + q / 2;
        if (block >= bk.b1)
            continue;
        const int64_t gcol = static_cast<int64_t>(bk.b0) * 64 + t * 128 + q * 32 + lane;
        const float bias = (!GATED && p.b1 != nullptr && gcol < p.O) ? __bfloat162float(p.b1[gcol]) : 0.0f;
        float v[CH], lin[CH];
#pragma unroll
        for (int i = 0; i < CH; ++i)
            lin[i] = 0.0f;
#pragma unroll 1
        for (int ch = 0; ch < NB / CH; ++ch) {
            tmem_chunk(tb + t * NB + ch * CH, v);
            if (GATED)
                tmem_chunk(tb + NB + ch * CH, lin);
            store_any<GATED>(p.act1, p.H, p.O, p.M, gcol, bias, v, lin, ch * CH, lane);
        }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0)
        ptx::mbar_arrive(ptx::smem_u32(&aux.tmem_empty[buf]));
    bool fenced = false;
#pragma unroll 1
    for (int t = 0; t < ntile; ++t) {
        const int32_t block = bk.b0 + 2 * t + q / 2;
        if (block >= bk.b1)
            continue;
        if (!fenced) {
            ptx::fence_proxy_async_global();
            __syncwarp();   // the warp's stores, then one release by lane 0 per block
            fenced = true;
        }
        if (lane == 0)
            ptx::st_release_gpu(p.flags + block * 2 + (q & 1), aux.epoch);
    }
}

// Per layer: drain every run as its accumulator completes (phase 1), then sum
// this CTA's shares of the split slices (phase 2).  A CTA stores all of its
// parts before it waits on anyone else's, so the waits cannot form a chain.
template <int NB, bool GLU, bool W2>
__device__ void run_epilogue(const Params& p, Aux& aux, const WaitCtx& w, uint8_t* ring, uint32_t tmem_base, int warp,
                             int lane)
{
    const int q = warp & 3;   // tensor-memory lanes 32q .. 32q + 31
    const Plan& pl = p.plan;
    uint32_t iter = 0, xphase = 0;
    for (int layer = 0; layer < 2; ++layer) {
        if (layer == 0 && pl.win) {
            const Blocks bk = blocks_of(pl);
            if (bk.b1 <= bk.b0)
                continue;
            const uint32_t buf = iter % Geo<NB>::NBUF;
            if (!wait_mbar(w, ptx::smem_u32(&aux.tmem_full[buf]), (iter / Geo<NB>::NBUF) & 1u, SITE_TMEM_FULL))
                return;
            ptx::tc_fence_after();
            drain_window<NB, GLU, W2>(p, aux, tmem_base, bk, buf, q, lane);
            ++iter;
            continue;
        }
        const Range r = range_of(pl, layer);
        for (int64_t u = r.u0; u < r.u1; ++u) {
            if (!run_last(r, u))
                continue;
            const uint32_t buf = iter % Geo<NB>::NBUF;
            if (!wait_mbar(w, ptx::smem_u32(&aux.tmem_full[buf]), (iter / Geo<NB>::NBUF) & 1u, SITE_TMEM_FULL))
                return;
            ptx::tc_fence_after();
            run_phase<NB, GLU, 1>(p, aux, w, ring, xphase, tmem_base, layer, u / r.kch, buf, q, lane);
            ++iter;
        }
        for (int64_t u = r.u0; u < r.u1; ++u) {
            if (!run_last(r, u))
                continue;
            if (!run_phase<NB, GLU, 2>(p, aux, w, ring, xphase, tmem_base, layer, u / r.kch, 0, q, lane))
                return;
        }
    }
}

template <int NB, bool GLU, bool W2>
__global__ void __launch_bounds__(NUM_THREADS, 1) wstream_kernel(const __grid_constant__ Params p)
{
    using Gm = Geo<NB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Aux& aux = *reinterpret_cast<Aux*>(stages + Gm::RING);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MAX_STAGES; ++s) {
            ptx::mbar_init(ptx::smem_u32(&aux.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.empty[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.full1[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.empty1[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&aux.tmem_full[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.tmem_empty[b]), EPI_WARPS);
        }
        ptx::mbar_init(ptx::smem_u32(&aux.drain), 1);
        for (int q = 0; q < EPI_WARPS; ++q)
            ptx::mbar_init(ptx::smem_u32(&aux.xfer[q]), 1);
        aux.abort = 0u;
        // device-side epoch: every CTA reads it before any can finish
        aux.epoch = *reinterpret_cast<volatile uint32_t*>(&p.ctrl->epoch) + 1u;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&p.map_w[0]);
        ptx::prefetch_tmap(&p.map_w[1]);
        ptx::prefetch_tmap(&p.map_x[0]);
        ptx::prefetch_tmap(&p.map_x[1]);
        if (GLU)
            ptx::prefetch_tmap(&p.map_w3);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&aux.tmem_base), Gm::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = aux.tmem_base;
    const WaitCtx w{&aux.abort, p.ctrl, p.wait_limit_ns, 0u};

    if (warp == 0) {
        run_producer<NB, GLU, W2>(p, aux, stages, w, lane);
    } else if (warp == 1) {
        if (lane == 0)
            run_mma<NB, GLU, W2>(p, aux, stages, w, tmem_base);
    } else {
        run_epilogue<NB, GLU, W2>(p, aux, w, stages, tmem_base, warp, lane);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, Gm::TMEM_COLS);
    }
    if (threadIdx.x == 0) {
        // The last CTA out publishes this launch's epoch.
        __threadfence();
        if (atomicAdd(&p.ctrl->ddone, 1u) == gridDim.x - 1) {
            p.ctrl->ddone = 0u;
            p.ctrl->epoch = aux.epoch;
            __threadfence();
        }
    }
}

}  // namespace wstream

namespace {

template <int NB, bool GLU, bool W2>
int launch_instance(const wstream::Params& p, cudaStream_t s)
{
    using Gm = wstream::Geo<NB>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(wstream::wstream_kernel<NB, GLU, W2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Gm::SMEM) != cudaSuccess)
            return -1;
        attr_set = true;
    }
    wstream::wstream_kernel<NB, GLU, W2><<<p.plan.grid, wstream::NUM_THREADS, Gm::SMEM, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_wstream(const wstream::Params& p, cudaStream_t s)
{
    if (p.plan.rows == 32)
        return p.glu ? launch_instance<32, true, false>(p, s)
                     : (p.plan.win == 2 ? launch_instance<32, false, true>(p, s) : launch_instance<32, false, false>(p, s));
    if (p.plan.rows == 64)
        return p.glu ? launch_instance<64, true, false>(p, s)
                     : (p.plan.win == 2 ? launch_instance<64, false, true>(p, s) : launch_instance<64, false, false>(p, s));
    if (p.plan.rows == 128)
        return p.glu ? launch_instance<128, true, false>(p, s)
                     : (p.plan.win == 2 ? launch_instance<128, false, true>(p, s) : launch_instance<128, false, false>(p, s));
    if (p.plan.rows == 256)
        return p.glu ? launch_instance<256, true, false>(p, s)
                     : (p.plan.win == 2 ? launch_instance<256, false, true>(p, s) : launch_instance<256, false, false>(p, s));
    return -1;
}

}  // namespace tffn
