// wstream.cuh -- the medium-batch weight stream: both FFN layers as one
// persistent launch that reads every weight byte once, on the tcgen05 tensor
// cores with the weights as the MMA's M side ("swap-AB").
//
// From 33 to 256 rows the FFN is still bound by the weight bytes (2 M FLOP per
// weight byte pair: M below the ~287 FLOP/byte ridge of a GB300), but the
// row-band engine has too few tiles to fill the GPU and mma.sync has too
// little throughput to keep up with HBM.  A 128-column tile of W (MN-major)
// is the A operand (M = 128) of an MMA, the K chunk of X or H (NB token rows,
// K-major) its B operand (N = NB), and the products accumulate in tensor
// memory, one lane per output column and one column per token.
//
// Layer 1 has many output columns and a short K, so it is not split: each
// CTA owns one or two (up to four) 64-column hidden blocks and computes a
// window of 128 (256) columns over all of K (Plan::win; the window's blocks
// it does not own are its neighbour's, computed and dropped).  Its H is
// final when the CTA's stream ends; the owning warps store it and stamp one
// ready word per block.
//
// Layer 2 has few output columns and a long K: a unit is KC = 64 rows of K
// for a slice of 256 output columns (two tiles sharing the H chunk), units
// spread over the CTAs as contiguous ranges (Stream-K, equal weight bytes per
// CTA).  A slice split across CTAs leaves fp32 partial sums in fixed places;
// once the slice's arrival counter shows every part ("Kernel fusion and
// tensor parallelism", section "Step 1": per-tile counters complete the
// tile), each contributing CTA sums its share of the slice's rows over all
// parts in part order, so the result does not depend on timing.  A layer-2
// range loads its first W2 stages, then waits for the H blocks it reads.
// (Hidden widths past four blocks per CTA run layer 1 the same way as layer
// 2, with ready words per H slice.)
//
// Gated layer 1 (H = act(X W1) * (X W3)): the window's two tiles are the
// same 128 columns of W1 and of W3, so the two accumulators hold the gate and
// the linear product and one thread has both values of its column.
//
// CTA layout (192 threads): warp 0 issues the TMA copies; warp 1 allocates
// tensor memory and one of its threads issues the MMAs; warps 2-5 drain the
// accumulators (warp w reads tensor-memory lanes 32 (w % 4) .. + 31).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstddef>
#include <cstdint>

#include "common.cuh"

namespace tffn {
namespace wstream {

constexpr int SLICE = 128;              // output columns of one MMA (its M); a unit has two
constexpr int KC = 64;                  // K rows per unit: one 128-byte swizzle row of B
constexpr int W_BOX = 64 * KC * 2;      // 8 KiB: 64 columns x KC rows of W
constexpr int EPI_WARPS = 4;
constexpr int NUM_THREADS = 32 * (2 + EPI_WARPS);
constexpr int MAX_STAGES = 8;
constexpr int MAX_ROWS = 256;           // rows (tokens) handled by this path
constexpr int MAX_GRID = 256;           // CTAs of one launch (one per SM)

// Geometry of the instance for at most NB token rows (NB a multiple of 32, up
// to 256).  Every unit carries two 128-column W tiles (four boxes, 32 KiB):
// the two halves of a 256-column output slice, or for the gated layer 1 the
// same 128 columns of W1 and W3; with the NB x KC tile of X or H this is a
// stage, and as many stages as fit 200 KiB are in flight (the weight bytes in
// flight per SM set the streaming rate).  A run's accumulator is two NB-column
// blocks of tensor memory; two of them (double buffering) up to NB = 128, one
// at NB = 256.
template <int NB>
struct Geo {
    static constexpr int W_BYTES = 4 * W_BOX;
    static constexpr int X_BYTES = NB * KC * 2;
    static constexpr int STAGE = W_BYTES + X_BYTES;
    static constexpr int NST0 = (200 * 1024) / STAGE;
    static constexpr int NST = NST0 > MAX_STAGES ? MAX_STAGES : NST0;
    // Window layer 1 (see Plan::win): a dense stage is one 128-column tile
    // and the X tile, in a ring of its own geometry over the same memory.
    static constexpr int STAGE1 = 2 * W_BOX + X_BYTES;
    static constexpr int NST1_0 = (200 * 1024) / STAGE1;
    static constexpr int NST1 = NST1_0 > MAX_STAGES ? MAX_STAGES : NST1_0;
    static constexpr int RING = NST * STAGE > NST1 * STAGE1 ? NST * STAGE : NST1 * STAGE1;
    static constexpr int ACC_COLS = 2 * NB;
    static constexpr int NBUF = 2 * ACC_COLS <= 512 ? 2 : 1;
    static constexpr int TMEM_COLS = NBUF * ACC_COLS;
    static constexpr int AUX = 1024;
    static constexpr int SMEM = RING + AUX + 1024;
    // At the end of layer 2 the ring is idle; each epilogue warp then loads
    // the parts it sums into its quarter of it (whole 2 KiB segments).
    static constexpr int WREG = (RING / EPI_WARPS) & ~2047;
    static constexpr int WSEGS = WREG / 2048;
    static_assert(SMEM <= 232448, "shared memory");
    static_assert(STAGE1 % 1024 == 0, "window stages stay 1024-byte aligned");
    static_assert(NB % 32 == 0 && NB <= 256, "token rows");
    static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "tensor-memory allocation");
    static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
};

// Token rows of the instance that serves M rows.
inline int stream_rows(int64_t M)
{
    return M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256));
}

struct Plan {
    int32_t grid;
    int32_t rows;           // NB of the instance
    // Window layer 1: CTA c owns the 64-column hidden blocks
    // [c * nblk / grid, (c + 1) * nblk / grid) (one or two) and computes them
    // over the whole of K as one 128-column tile (the second block of a
    // one-block CTA is its neighbour's, computed and dropped): no split
    // slices, so H is final when a CTA's stream ends.  win = 1 when every
    // CTA owns at most two blocks (hidden width up to 128 x CTAs); win = 2
    // (dense) up to four, the window then two 128-column tiles (256
    // columns, the stage geometry of layer 2); otherwise (win = 0) layer 1
    // is a Stream-K over 256-column slices like layer 2.
    int32_t win;
    int32_t nblk;           // 64-column hidden blocks (window layer 1)
    int32_t h_cols;         // hidden columns of a layer-1 slice: 256, or 128 gated
    int32_t slices[2];      // output slices per layer (256 columns; gated layer 1: 128)
    int32_t kch[2];         // K chunks (KC rows) per slice
    int64_t units[2];       // slices * kch
    int32_t maxp[2];        // most CTAs sharing one slice
    int64_t part_off[2];    // float offset of each layer's partial sums
    size_t partial_bytes;
    uint8_t split[2][MAX_GRID];   // per CTA: its split slices (shared with other CTAs) per layer
};

// CTA that owns unit u when U units are spread over G CTAs (U >= G).
__host__ __device__ inline int64_t owner_of(int64_t u, int64_t U, int64_t G)
{
    return ((u + 1) * G + U - 1) / U - 1;
}

__host__ __device__ inline int64_t range_start(int64_t c, int64_t U, int64_t G)
{
    return c * U / G;
}

// Floats of one part's partial sums: two halves x 128 columns x NB rows.
__host__ __device__ inline int64_t part_floats(int rows)
{
    return static_cast<int64_t>(2) * SLICE * rows;
}

// Layout of one part, by epilogue warp: warp q's 32 columns of half a, rows
// [16 ch, 16 ch + 16), form one 2 KiB segment at float offset seg_off(q, a,
// ch); in it, float4 i of lane l (rows 4i .. 4i+3 of column 32 q + l) sits
// at float (i * 32 + l) * 4.  A warp's data of one item is contiguous, so a
// warp can fetch it with one bulk copy; a warp store instruction covers 512
// contiguous bytes.
constexpr int SEG_FLOATS = 512;

template <int NB>
__host__ __device__ inline int64_t seg_off(int q, int a, int ch)
{
    return ((static_cast<int64_t>(q) * 2 + a) * (NB / 16) + ch) * SEG_FLOATS;
}

// grid is the CTA count the caller wants; it is lowered so that every CTA
// owns at least one unit of each layer.
inline Plan make_plan(int64_t M, int64_t N, int64_t O, int64_t P, int grid, bool glu)
{
    Plan pl{};
    pl.rows = stream_rows(M);
    pl.h_cols = glu ? SLICE : 2 * SLICE;
    pl.slices[0] = static_cast<int32_t>((O + pl.h_cols - 1) / pl.h_cols);
    pl.kch[0] = static_cast<int32_t>((N + KC - 1) / KC);
    pl.slices[1] = static_cast<int32_t>((P + 2 * SLICE - 1) / (2 * SLICE));
    pl.kch[1] = static_cast<int32_t>((O + KC - 1) / KC);
    int64_t g = grid < MAX_GRID ? grid : MAX_GRID;
    for (int l = 0; l < 2; ++l)
        pl.units[l] = static_cast<int64_t>(pl.slices[l]) * pl.kch[l];
    if (pl.units[1] < g)
        g = pl.units[1];
    if (g < 1)
        g = 1;
    pl.nblk = static_cast<int32_t>((O + 63) / 64);
    pl.win = pl.nblk <= 2 * g ? 1 : ((!glu && pl.nblk <= 4 * g) ? 2 : 0);
    if (!pl.win && pl.units[0] < g)
        g = pl.units[0];
    pl.grid = static_cast<int32_t>(g);
    int64_t off = 0;
    if (pl.win) {
        // the window layer 1 is never split: one part per hidden block
        pl.maxp[0] = 1;
        pl.part_off[0] = 0;
    }
    for (int l = pl.win ? 1 : 0; l < 2; ++l) {
        int32_t maxp = 1;
        for (int64_t s = 0; s < pl.slices[l]; ++s) {
            const int64_t a = owner_of(s * pl.kch[l], pl.units[l], g);
            const int64_t b = owner_of((s + 1) * pl.kch[l] - 1, pl.units[l], g);
            if (b - a + 1 > maxp)
                maxp = static_cast<int32_t>(b - a + 1);
        }
        pl.maxp[l] = maxp;
        pl.part_off[l] = off;
        if (maxp > 1)
            off += static_cast<int64_t>(pl.slices[l]) * maxp * part_floats(pl.rows);
    }
    pl.partial_bytes = static_cast<size_t>(off) * 4;
    for (int l = pl.win ? 1 : 0; l < 2; ++l) {
        const int64_t U = pl.units[l], kch = pl.kch[l];
        for (int64_t c = 0; c < g; ++c) {
            const int64_t u0 = range_start(c, U, g), u1 = range_start(c + 1, U, g);
            int n = 0;
            for (int64_t sl = u0 / kch; sl <= (u1 - 1) / kch; ++sl)
                n += owner_of(sl * kch, U, g) != owner_of((sl + 1) * kch - 1, U, g) ? 1 : 0;
            pl.split[l][c] = static_cast<uint8_t>(n < 255 ? n : 255);
        }
    }
    return pl;
}

struct Params {
    CUtensorMap map_w[2];      // W1 {O, N}, W2 {P, O}; box {64, KC}
    CUtensorMap map_w3;        // gated form: W3 {O, N}; box {64, KC}
    CUtensorMap map_x[2];      // X {N, M}, H {O, M}; box {64, NB} (rows past M read as zeros)
    const __nv_bfloat16* b1;
    const __nv_bfloat16* b2;
    __nv_bfloat16* Y;          // [M x P]
    __nv_bfloat16* H;          // [M x O]
    float* partial;
    uint32_t* counters;        // arrival counters [slices0 * 4] then [slices1 * 4] (one per epilogue
                               // warp), then the done counters in the same layout
    uint32_t* flags;           // H ready (= epoch): [slices0 * 4], one word per slice and epilogue warp;
                               // window layer 1: [nblk * 2], one per 64-column block and warp
    DevCtrl* ctrl;
    int32_t M, N, O, P;
    int32_t act1, act2;
    int32_t glu;
    uint64_t wait_limit_ns;
    Plan plan;
};

}  // namespace wstream
}  // namespace tffn
