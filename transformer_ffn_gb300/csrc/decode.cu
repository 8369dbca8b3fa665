// decode.cu -- the weight-streaming small-M FFN kernel (see decode.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "decode.cuh"
#include "launch.h"

namespace tffn {
namespace decode {

static_assert(SLICE == KC, "a layer-2 unit reads one dense (or two gated) layer-1 slices of H");

struct Aux {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint32_t abort;
    uint32_t epoch;     // this launch's ready-flag value (control block's + 1)
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled
// box (rows of 128 bytes; chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

template <int MT>
struct Acc {
    float c[MT][4][4];   // [m tile][n8 tile][fragment]
};

template <int MT>
__device__ __forceinline__ void zero(Acc<MT>& a)
{
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                a.c[m][n][i] = 0.0f;
}

// One KC x SLICE unit: this warp's 32 columns, all K rows of the stage.  The
// fragments of four k-steps are loaded first and the MMAs issued after, so the
// shared-memory latency of the loads overlaps instead of sitting in front of
// every MMA.
// Gated (GLU): n8 tiles 0-1 come from the W1 box and 2-3 from the W3 box,
// the same 16 columns (chunks 2cw, 2cw+1) of each.
template <int MT, bool GLU>
__device__ __forceinline__ void compute_stage(Acc<MT>& acc, uint32_t w_base, uint32_t a_base, int cw, int lane)
{
    const uint32_t wbox_dense = w_base + static_cast<uint32_t>(cw >> 1) * W_BOX_BYTES;
    const uint32_t cb_chunk = GLU ? static_cast<uint32_t>(cw) * 2 : static_cast<uint32_t>(cw & 1) * 4;
    const uint32_t j = static_cast<uint32_t>(lane >> 3);
    const uint32_t r = static_cast<uint32_t>(lane & 7);
    constexpr int KB = Geo<MT>::KB;
#pragma unroll
    for (int kb0 = 0; kb0 < KC / 16; kb0 += KB) {
        uint32_t a[KB][MT][4];
        uint32_t b[KB][2][4];
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
            const int ks = kb0 + kk;
            const uint32_t abox = a_base + static_cast<uint32_t>(ks >> 2) * Geo<MT>::A_BOX;
            const uint32_t kchunk = static_cast<uint32_t>((ks & 3) * 2) + (j >> 1);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint32_t row = static_cast<uint32_t>(m * 16) + (j & 1u) * 8u + r;
                ldsm_x4(abox + sw128(row, kchunk), a[kk][m][0], a[kk][m][1], a[kk][m][2], a[kk][m][3]);
            }
            const uint32_t krow = static_cast<uint32_t>(ks * 16) + (j & 1u) * 8u + r;
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const uint32_t wbox = GLU ? w_base + static_cast<uint32_t>(pr) * W_BOX_BYTES : wbox_dense;
                const uint32_t nchunk = cb_chunk + (GLU ? 0u : static_cast<uint32_t>(pr * 2)) + (j >> 1);
                ldsm_x4_t(wbox + sw128(krow, nchunk), b[kk][pr][0], b[kk][pr][1], b[kk][pr][2], b[kk][pr][3]);
            }
        }
#pragma unroll
        for (int kk = 0; kk < KB; ++kk)
#pragma unroll
            for (int pr = 0; pr < 2; ++pr)
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    mma_bf16_16816(acc.c[m][pr * 2 + 0], a[kk][m][0], a[kk][m][1], a[kk][m][2], a[kk][m][3],
                                   b[kk][pr][0], b[kk][pr][1]);
                    mma_bf16_16816(acc.c[m][pr * 2 + 1], a[kk][m][0], a[kk][m][1], a[kk][m][2], a[kk][m][3],
                                   b[kk][pr][2], b[kk][pr][3]);
                }
    }
}

// Gated window layer 1: accumulators of this warp's 32 hidden columns, n8
// tiles 0-3 the gate (X W1) and 4-7 the linear product (X W3) of the same
// columns.
template <int MT>
struct AccW {
    float c[MT][8][4];
};

// One KC1-deep stage of the window: W1 boxes 0-1 (128 columns) then W3 boxes
// 2-3, each KC1 rows x 64 columns, 128-byte swizzled; warp cw takes columns
// [32cw, 32cw + 32) of W1 and of W3.
template <int MT>
__device__ __forceinline__ void compute_stage_win(AccW<MT>& acc, uint32_t w_base, uint32_t a_base, int cw, int lane)
{
    constexpr uint32_t BOX = KC1 * 128;
    const uint32_t g_box = w_base + static_cast<uint32_t>(cw >> 1) * BOX;
    const uint32_t l_box = g_box + 2 * BOX;
    const uint32_t cb = static_cast<uint32_t>(cw & 1) * 4;
    const uint32_t j = static_cast<uint32_t>(lane >> 3);
    const uint32_t r = static_cast<uint32_t>(lane & 7);
    constexpr int KB = Geo<MT>::KB;
#pragma unroll
    for (int kb0 = 0; kb0 < KC1 / 16; kb0 += KB) {
        uint32_t a[KB][MT][4];
        uint32_t b[KB][4][4];   // gate cols 0-15, gate 16-31, linear 0-15, linear 16-31
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
            const int ks = kb0 + kk;
            const uint32_t kchunk = static_cast<uint32_t>((ks & 3) * 2) + (j >> 1);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint32_t row = static_cast<uint32_t>(m * 16) + (j & 1u) * 8u + r;
                ldsm_x4(a_base + sw128(row, kchunk), a[kk][m][0], a[kk][m][1], a[kk][m][2], a[kk][m][3]);
            }
            const uint32_t krow = static_cast<uint32_t>(ks * 16) + (j & 1u) * 8u + r;
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const uint32_t nchunk = cb + static_cast<uint32_t>(pr * 2) + (j >> 1);
                ldsm_x4_t(g_box + sw128(krow, nchunk), b[kk][pr][0], b[kk][pr][1], b[kk][pr][2], b[kk][pr][3]);
                ldsm_x4_t(l_box + sw128(krow, nchunk), b[kk][2 + pr][0], b[kk][2 + pr][1], b[kk][2 + pr][2],
                          b[kk][2 + pr][3]);
            }
        }
#pragma unroll
        for (int kk = 0; kk < KB; ++kk)
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    mma_bf16_16816(acc.c[m][t * 2 + 0], a[kk][m][0], a[kk][m][1], a[kk][m][2], a[kk][m][3],
                                   b[kk][t][0], b[kk][t][1]);
                    mma_bf16_16816(acc.c[m][t * 2 + 1], a[kk][m][0], a[kk][m][1], a[kk][m][2], a[kk][m][3],
                                   b[kk][t][2], b[kk][t][3]);
                }
    }
}

// The window's H: warp cw's 32 columns lie in block b0 + cw / 2; when the CTA
// owns that block the warp writes act(gate) * linear (bf16) and stamps the
// block's word for its half.
template <int MT>
__device__ void flush_win(const Params& p, int32_t b0, int32_t b1, const AccW<MT>& acc, int cw, int lane,
                          uint32_t epoch)
{
    const int32_t block = b0 + (cw >> 1);
    if (block >= b1)
        return;
    const int g = lane >> 2, q = lane & 3;
    const int M = p.M;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
        const int col = b0 * 64 + cw * 32 + n * 8 + 2 * q;
        if (col >= p.O)
            continue;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int r0 = m * 16 + g, r1 = r0 + 8;
            if (r0 < M)
                *reinterpret_cast<uint32_t*>(p.H + static_cast<int64_t>(r0) * p.O + col) =
                    pack_bf16x2(act_apply(p.act1, acc.c[m][n][0]) * acc.c[m][n + 4][0],
                                act_apply(p.act1, acc.c[m][n][1]) * acc.c[m][n + 4][1]);
            if (r1 < M)
                *reinterpret_cast<uint32_t*>(p.H + static_cast<int64_t>(r1) * p.O + col) =
                    pack_bf16x2(act_apply(p.act1, acc.c[m][n][2]) * acc.c[m][n + 4][2],
                                act_apply(p.act1, acc.c[m][n][3]) * acc.c[m][n + 4][3]);
        }
    }
    ptx::fence_proxy_async_global();
    __syncwarp();   // the warp's stores, then one release by lane 0
    if (lane == 0)
        ptx::st_release_gpu(p.flags + block * 2 + (cw & 1), epoch);
}

// Adds parts [1, nparts) of this warp's columns, in part order, to acc (which
// holds part 0); F parts' loads are in flight at a time.
template <int MT, int F>
__device__ __forceinline__ void add_parts(Acc<MT>& acc, const float* base, int nparts, int cw, int lane, int M)
{
    const int g = lane >> 2, q = lane & 3;
#pragma unroll 1
    for (int pp = 1; pp < nparts; pp += F) {
        float2 v[F][MT][4][2];
#pragma unroll
        for (int j = 0; j < F; ++j) {
            const float* src = base + static_cast<int64_t>(pp + j) * Geo<MT>::ROWS * SLICE;
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    const int col = cw * 32 + n * 8 + 2 * q;
                    const int r0 = m * 16 + g, r1 = r0 + 8;
                    const bool in = pp + j < nparts;
                    v[j][m][n][0] = (in && r0 < M) ? __ldcg(reinterpret_cast<const float2*>(src + r0 * SLICE + col))
                                                   : make_float2(0.f, 0.f);
                    v[j][m][n][1] = (in && r1 < M) ? __ldcg(reinterpret_cast<const float2*>(src + r1 * SLICE + col))
                                                   : make_float2(0.f, 0.f);
                }
        }
#pragma unroll
        for (int j = 0; j < F; ++j) {
            if (pp + j >= nparts)
                break;
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    acc.c[m][n][0] += v[j][m][n][0].x;
                    acc.c[m][n][1] += v[j][m][n][0].y;
                    acc.c[m][n][2] += v[j][m][n][1].x;
                    acc.c[m][n][3] += v[j][m][n][1].y;
                }
        }
    }
}

// Finish this warp's 32 columns of one slice: direct epilogue when one CTA
// owns the whole K range.  A split slice's parts are its CTAs' runs in CTA
// order; part 0 is the run that ends its CTA's range (the slice continues in
// the next CTA), so it is normally finished last, and its CTA reduces: it
// waits until the slice's counter shows the other nparts - 1 parts, adds them
// in part order to its own registers, and writes the output.  Every other
// part stores its partial and leaves the counter increment in `pending`: the
// caller publishes it (one release by lane 0) after its next stage, when the
// stores have drained, instead of stalling the warp on them now.
// Returns false on abort or timeout.
template <int MT>
__device__ bool flush(const Params& p, const WaitCtx& w, int layer, int64_t slice, Acc<MT>& acc, int cw, int lane,
                      uint32_t epoch, uint32_t*& pending)
{
    const Plan& pl = p.plan;
    const int64_t U = pl.units[layer], G = pl.grid, kch = pl.kch[layer];
    const int64_t first = owner_of(slice * kch, U, G);
    const int64_t last = owner_of((slice + 1) * kch - 1, U, G);
    const int nparts = static_cast<int>(last - first + 1);
    const int part = static_cast<int>(blockIdx.x - first);
    const int g = lane >> 2, q = lane & 3;
    const int M = p.M;

    if (nparts > 1) {
        const float* base = p.partial + pl.part_off[layer] +
                            (static_cast<int64_t>(slice) * pl.maxp[layer]) * Geo<MT>::ROWS * SLICE;
        uint32_t* cnt = p.counters + (layer == 0 ? 0 : pl.slices[0] * 4) + slice * 4 + cw;
        if (part != 0) {
            float* mine = const_cast<float*>(base) + static_cast<int64_t>(part) * Geo<MT>::ROWS * SLICE;
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    const int col = cw * 32 + n * 8 + 2 * q;
                    const int r0 = m * 16 + g, r1 = r0 + 8;
                    if (r0 < M)
                        *reinterpret_cast<float2*>(mine + r0 * SLICE + col) =
                            make_float2(acc.c[m][n][0], acc.c[m][n][1]);
                    if (r1 < M)
                        *reinterpret_cast<float2*>(mine + r1 * SLICE + col) =
                            make_float2(acc.c[m][n][2], acc.c[m][n][3]);
                }
            pending = cnt;
            return true;
        }
        bool ok = true;
        if (lane == 0)
            ok = wait_flag(w, cnt, static_cast<uint32_t>(nparts - 1), SITE_PARTS, static_cast<uint32_t>(slice));
        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0)
            return false;
        __syncwarp();   // lane 0's acquire covers the warp's reads of the parts
        add_parts<MT, (MT == 1 ? 4 : (MT == 2 ? 2 : 1))>(acc, base, nparts, cw, lane, M);
        if (lane == 0)
            *cnt = 0u;   // every other part has arrived: ready for the next call
    }

    if (layer == 0 && p.glu) {
        // Gated: H = act(gate) * lin for this warp's 16 hidden columns.
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const int col = static_cast<int>(slice) * (SLICE / 2) + cw * 16 + n * 8 + 2 * q;
            if (col >= p.O)
                continue;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const int r0 = m * 16 + g, r1 = r0 + 8;
                if (r0 < M)
                    *reinterpret_cast<uint32_t*>(p.H + static_cast<int64_t>(r0) * p.O + col) =
                        pack_bf16x2(act_apply(p.act1, acc.c[m][n][0]) * acc.c[m][n + 2][0],
                                    act_apply(p.act1, acc.c[m][n][1]) * acc.c[m][n + 2][1]);
                if (r1 < M)
                    *reinterpret_cast<uint32_t*>(p.H + static_cast<int64_t>(r1) * p.O + col) =
                        pack_bf16x2(act_apply(p.act1, acc.c[m][n][2]) * acc.c[m][n + 2][2],
                                    act_apply(p.act1, acc.c[m][n][3]) * acc.c[m][n + 2][3]);
            }
        }
        ptx::fence_proxy_async_global();
        __syncwarp();   // the warp's stores, then one release by lane 0
        if (lane == 0)
            ptx::st_release_gpu(p.flags + slice * CONSUMER_WARPS + cw, epoch);
        return true;
    }

    // Epilogue: bias, activation, bf16.
    const __nv_bfloat16* bias = layer == 0 ? p.b1 : p.b2;
    const int act = layer == 0 ? p.act1 : p.act2;
    const int ncols = layer == 0 ? p.O : p.P;
    __nv_bfloat16* out = layer == 0 ? p.H : p.Y;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
        const int col = static_cast<int>(slice) * SLICE + cw * 32 + n * 8 + 2 * q;
        if (col >= ncols)
            continue;
        float b0 = 0.f, b1 = 0.f;
        if (bias) {
            const uint32_t bb = *reinterpret_cast<const uint32_t*>(bias + col);
            b0 = bf16_lo(bb);
            b1 = bf16_hi(bb);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int r0 = m * 16 + g, r1 = r0 + 8;
            if (r0 < M)
                *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(r0) * ncols + col) =
                    pack_bf16x2(act_apply(act, acc.c[m][n][0] + b0), act_apply(act, acc.c[m][n][1] + b1));
            if (r1 < M)
                *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(r1) * ncols + col) =
                    pack_bf16x2(act_apply(act, acc.c[m][n][2] + b0), act_apply(act, acc.c[m][n][3] + b1));
        }
    }
    if (layer == 0) {
        // Publish this warp's quarter of the H slice: stamp its flag word with
        // the call's epoch (release, gpu scope).
        ptx::fence_proxy_async_global();
        __syncwarp();   // the warp's stores, then one release by lane 0
        if (lane == 0 && slice != p.skip_slice)
            ptx::st_release_gpu(p.flags + slice * CONSUMER_WARPS + cw, epoch);
    }
    return true;
}

// Wait, with the whole warp, until every layer-1 slice of H read by the
// cyclic window [k0, k0 + count) of kch layer-2 K chunks is ready (all four
// words equal the epoch; h_per_k slices per chunk).  Relaxed loads spread over
// the lanes, then an acquire fence in every lane: one pass over many flags
// instead of one serialised acquire per unit.
__device__ bool wait_h_window(const WaitCtx& w, const uint32_t* flags, uint32_t epoch, int64_t k0, int64_t count,
                              int64_t kch, int h_per_k, int64_t h_slices, bool win, int lane)
{
    const int nw = win ? 2 : CONSUMER_WARPS;   // ready words per slice (window: per block)
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        bool mine = true;
        for (int64_t i = lane; i < count * h_per_k && mine; i += 32) {
            const int64_t hs = ((k0 + i / h_per_k) % kch) * h_per_k + i % h_per_k;
            if (hs >= h_slices)
                continue;   // past the last hidden column: nothing to wait for
            const uint32_t* f = flags + hs * nw;
#pragma unroll
            for (int q = 0; q < CONSUMER_WARPS; ++q)
                if (q < nw) {
                    uint32_t v;
                    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f + q) : "memory");
                    mine = mine && (v == epoch);
                }
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

// Warp 0.  Layer 1 streams W1 and X; layer 2 first prefetches the W2 part of
// its first stages (W2 does not depend on H), then waits once for every H
// slice its unit range reads, then streams W2 and H.
template <int MT>
__device__ void run_producer(const Params& p, Aux& aux, uint8_t* stages, const WaitCtx& w, int lane)
{
    constexpr uint32_t A_BYTES = 2u * (16u * MT) * 64u * 2u;
    constexpr int STAGES = Geo<MT>::NST;
    constexpr int STAGE_BYTES = Geo<MT>::STAGE;
    const Plan& pl = p.plan;
    const int64_t G = pl.grid, c = blockIdx.x;
    uint32_t stage = 0, phase = 0;
    int32_t last_phase[STAGES];
    for (int s = 0; s < STAGES; ++s)
        last_phase[s] = -1;
    uint64_t evict_first = 0;
    if (lane == 0)
        evict_first = ptx::policy_evict_first();
    bool ok = true;

    auto issue_w = [&](int layer, int64_t slice, int64_t kc, uint32_t st) {
        const uint32_t fb = ptx::smem_u32(&aux.full[st]);
        const uint32_t sw = ptx::smem_u32(stages + st * STAGE_BYTES);
        if (layer == 0 && p.glu) {   // the same 64 hidden columns of W1 and of W3
            ptx::tma_load_2d_hint(sw, &p.map_w[0], fb, static_cast<int32_t>(slice * (SLICE / 2)),
                                  static_cast<int32_t>(kc * KC), evict_first);
            ptx::tma_load_2d_hint(sw + W_BOX_BYTES, &p.map_w3, fb, static_cast<int32_t>(slice * (SLICE / 2)),
                                  static_cast<int32_t>(kc * KC), evict_first);
            return;
        }
        ptx::tma_load_2d_hint(sw, &p.map_w[layer], fb, static_cast<int32_t>(slice * SLICE),
                              static_cast<int32_t>(kc * KC), evict_first);
        ptx::tma_load_2d_hint(sw + W_BOX_BYTES, &p.map_w[layer], fb, static_cast<int32_t>(slice * SLICE + 64),
                              static_cast<int32_t>(kc * KC), evict_first);
    };
    auto issue_a = [&](int layer, int64_t kc, uint32_t st) {
        const uint32_t fb = ptx::smem_u32(&aux.full[st]);
        const uint32_t sa = ptx::smem_u32(stages + st * STAGE_BYTES) + W_STAGE_BYTES;
        ptx::tma_load_2d(sa, &p.map_a[layer], fb, static_cast<int32_t>(kc * KC), 0);
        ptx::tma_load_2d(sa + Geo<MT>::A_BOX, &p.map_a[layer], fb, static_cast<int32_t>(kc * KC + 64), 0);
    };
    auto advance = [&]() {
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    };

    // ---- layer 1
    if (lane == 0 && pl.win) {
        // gated window: W1 and W3 boxes of the CTA's 128 hidden columns and
        // one A box per KC1-row chunk
        constexpr uint32_t BOX = KC1 * 128;
        constexpr uint32_t A1_BYTES = (16u * MT) * 64u * 2u;
        const int32_t b0 = static_cast<int32_t>(c * pl.nblk / G), b1 = static_cast<int32_t>((c + 1) * pl.nblk / G);
        if (b1 > b0) {
            const int32_t col0 = b0 * 64;
            for (int64_t kc = 0; kc < pl.kch[0]; ++kc) {
                ok = wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY);
                if (!ok)
                    break;
                const uint32_t fb = ptx::smem_u32(&aux.full[stage]);
                const uint32_t sw = ptx::smem_u32(stages + stage * STAGE_BYTES);
                const int32_t row = static_cast<int32_t>(kc * KC1);
                ptx::mbar_arrive_expect_tx(fb, 4 * BOX + A1_BYTES);
                ptx::tma_load_2d(sw, &p.map_w[0], fb, col0, row);
                ptx::tma_load_2d(sw + BOX, &p.map_w[0], fb, col0 + 64, row);
                ptx::tma_load_2d(sw + 2 * BOX, &p.map_w3, fb, col0, row);
                ptx::tma_load_2d(sw + 3 * BOX, &p.map_w3, fb, col0 + 64, row);
                ptx::tma_load_2d(sw + W_STAGE_BYTES, &p.map_a[0], fb, row, 0);
                last_phase[stage] = static_cast<int32_t>(phase);
                advance();
            }
        }
    } else if (lane == 0) {
        const int64_t U = pl.units[0], kch = pl.kch[0];
        const int64_t u0 = range_start(c, U, G), u1 = range_start(c + 1, U, G);
        for (int64_t u = u0; u < u1; ++u) {
            ok = wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY);
            if (!ok)
                break;
            ptx::mbar_arrive_expect_tx(ptx::smem_u32(&aux.full[stage]), W_STAGE_BYTES + A_BYTES);
            issue_w(0, u / kch, u % kch, stage);
            issue_a(0, u % kch, stage);
            last_phase[stage] = static_cast<int32_t>(phase);
            advance();
        }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;

    // ---- layer 2
    if (ok) {
        const int64_t U = pl.units[1], kch = pl.kch[1];
        const int64_t u0 = range_start(c, U, G), u1 = range_start(c + 1, U, G);
        const int64_t npre = (u1 - u0) < STAGES ? (u1 - u0) : STAGES;
        uint32_t pre_stage[STAGES];
        if (lane == 0) {
            for (int64_t i = 0; i < npre; ++i) {
                const int64_t u = u0 + i;
                ok = wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY);
                if (!ok)
                    break;
                ptx::mbar_arrive_expect_tx(ptx::smem_u32(&aux.full[stage]), W_STAGE_BYTES + A_BYTES);
                issue_w(1, u / kch, u % kch, stage);
                pre_stage[i] = stage;
                last_phase[stage] = static_cast<int32_t>(phase);
                advance();
            }
        }
        const int npre_done = __shfl_sync(0xffffffffu, ok ? static_cast<int>(npre) : -1, 0);
        if (npre_done >= 0) {
            const int64_t count = (u1 - u0) < kch ? (u1 - u0) : kch;
            const bool ready = wait_h_window(w, p.flags, aux.epoch, u0 % kch, count, kch, pl.h_per_k, pl.slices[0],
                                             pl.win != 0, lane);
            if (lane == 0) {
                ptx::fence_proxy_async_global();
                // the prefetched stages expect their H bytes: issue them even
                // after a failed wait so that every barrier completes
                for (int64_t i = 0; i < npre; ++i)
                    issue_a(1, (u0 + i) % kch, pre_stage[i]);
                if (ready) {
                    for (int64_t u = u0 + npre; u < u1; ++u) {
                        if (!wait_mbar(w, ptx::smem_u32(&aux.empty[stage]), phase ^ 1u, SITE_SMEM_EMPTY))
                            break;
                        ptx::mbar_arrive_expect_tx(ptx::smem_u32(&aux.full[stage]), W_STAGE_BYTES + A_BYTES);
                        issue_w(1, u / kch, u % kch, stage);
                        issue_a(1, u % kch, stage);
                        last_phase[stage] = static_cast<int32_t>(phase);
                        advance();
                    }
                }
            }
        }
    }

    // Exit: every copy issued by this warp has landed before the CTA leaves.
    if (lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
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

template <int MT>
__global__ void __launch_bounds__(NUM_THREADS, 1) decode_kernel(const __grid_constant__ Params p)
{
    constexpr int STAGES = Geo<MT>::NST;
    constexpr int STAGE_BYTES = Geo<MT>::STAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Aux& aux = *reinterpret_cast<Aux*>(stages + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const Plan& pl = p.plan;
    const int64_t G = pl.grid;
    const int64_t c = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_u32(&aux.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&aux.empty[s]), CONSUMER_WARPS);
        }
        aux.abort = 0u;
        // device-side epoch: every CTA reads it before any can finish
        aux.epoch = *reinterpret_cast<volatile uint32_t*>(&p.ctrl->epoch) + 1u;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    const WaitCtx w{&aux.abort, p.ctrl, p.wait_limit_ns};

    if (warp == 0) {
        run_producer<MT>(p, aux, stages, w, lane);
    } else {
        const int cw = warp - 1;
        uint32_t stage = 0, phase = 0;
        Acc<MT> acc;
        bool ok = true;
        uint32_t* pending = nullptr;   // a stored part whose counter increment is still to be published
        auto publish = [&]() {
            if (pending != nullptr) {
                __syncwarp();   // the warp's partial stores, then one release by lane 0
                if (lane == 0)
                    ptx::red_release_add_gpu(pending, 1u);
                pending = nullptr;
            }
        };
        for (int layer = 0; layer < 2 && ok; ++layer) {
            if constexpr (MT <= 2) {
                if (layer == 0 && pl.win) {
                    const int32_t b0 = static_cast<int32_t>(c * pl.nblk / G);
                    const int32_t b1 = static_cast<int32_t>((c + 1) * pl.nblk / G);
                    if (b1 <= b0)
                        continue;
                    AccW<MT> aw;
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int n = 0; n < 8; ++n)
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                aw.c[m][n][i] = 0.0f;
                    for (int64_t kc = 0; kc < pl.kch[0]; ++kc) {
                        ok = wait_mbar(w, ptx::smem_u32(&aux.full[stage]), phase, SITE_STAGE);
                        if (!ok)
                            break;
                        const uint32_t sw = ptx::smem_u32(stages + stage * STAGE_BYTES);
                        compute_stage_win<MT>(aw, sw, sw + W_STAGE_BYTES, cw, lane);
                        __syncwarp();
                        if (lane == 0)
                            ptx::mbar_arrive(ptx::smem_u32(&aux.empty[stage]));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok)
                        flush_win<MT>(p, b0, b1, aw, cw, lane, aux.epoch);
                    continue;
                }
            }
            const int64_t U = pl.units[layer], kch = pl.kch[layer];
            const int64_t u0 = range_start(c, U, G), u1 = range_start(c + 1, U, G);
            int64_t cur = -1;
            for (int64_t u = u0; u < u1; ++u) {
                const int64_t slice = u / kch;
                if (slice != cur) {
                    if (cur >= 0 && !flush<MT>(p, w, layer, cur, acc, cw, lane, aux.epoch, pending)) {
                        ok = false;
                        break;
                    }
                    zero(acc);
                    cur = slice;
                }
                ok = wait_mbar(w, ptx::smem_u32(&aux.full[stage]), phase, SITE_STAGE);
                if (!ok)
                    break;
                const uint32_t sw = ptx::smem_u32(stages + stage * STAGE_BYTES);
                if (layer == 0 && p.glu)
                    compute_stage<MT, true>(acc, sw, sw + W_STAGE_BYTES, cw, lane);
                else
                    compute_stage<MT, false>(acc, sw, sw + W_STAGE_BYTES, cw, lane);
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(ptx::smem_u32(&aux.empty[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                publish();   // a part flushed before this stage: its stores have had a stage to drain
            }
            if (ok && cur >= 0)
                ok = flush<MT>(p, w, layer, cur, acc, cw, lane, aux.epoch, pending);
            publish();
        }
    }
    __syncwarp();
    __syncthreads();
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

}  // namespace decode

namespace {

template <int MT>
int launch_decode_mt(const decode::Params& p, cudaStream_t s)
{
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(decode::decode_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 decode::Geo<MT>::SMEM) != cudaSuccess)
            return -1;
        attr_set = true;
    }
    decode::decode_kernel<MT><<<p.plan.grid, decode::NUM_THREADS, decode::Geo<MT>::SMEM, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_decode(const decode::Params& p, int grid, cudaStream_t s)
{
    (void)grid;
    if (p.M <= 16)
        return launch_decode_mt<1>(p, s);
    if (p.M <= 32)
        return launch_decode_mt<2>(p, s);
    return launch_decode_mt<4>(p, s);
}

}  // namespace tffn
