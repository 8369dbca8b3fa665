// decode.cuh -- the small-M (decode) path: both layers of the FFN as one
// persistent launch that streams the weights from HBM exactly once.
//
// At M <= 64 rows the FFN is bound by reading W1 and W2 ("kernel fusion"
// page, section "Complexity and constants": a memory-bound kernel takes the
// bytes it moves divided by the achievable HBM bandwidth, and needs 16-byte
// accesses to get there).  Work is cut into units of SLICE output columns x KC
// rows of K; CTA c of G owns the contiguous unit range [c*U/G, (c+1)*U/G) of
// each layer (Stream-K style: every CTA gets the same amount of weight bytes).
// A slice whose K range is split across CTAs is finished by the CTA holding
// its part 0 (the run that ends that CTA's range, normally the last part to
// be done): once the slice's counter shows the other parts it adds them in
// part order to its own, so the result does not depend on arrival order
// ("Kernel fusion and tensor parallelism", section "Step 1": a per-tile
// counter completes the tile; the accumulation of partial tiles with
// completion flags that Stream-K uses).  A finished layer-1 slice of H
// publishes a ready flag; layer-2 units wait on the flags of the H slices
// they read.
//
// Gated FFN (H = act(X W1) * (X W3)), up to 32 rows: layer 1 is a window
// instead (Plan::win): each CTA owns one or two 64-column hidden blocks and
// streams 128 adjacent columns of W1 and of W3 over all of K, each consumer
// warp taking 32 columns of each, so every thread ends with the gate and
// linear fragments of the same H elements; no split, one ready word per block
// and owning warp.  A layer-2 K chunk reads two 64-column blocks of H.
//
// Layout per CTA: warp 0 issues TMA copies (W tile [KC x SLICE] as two
// 128-byte-swizzled boxes, plus the [rows x KC] tile of X or H); warps 1..4
// each own 32 of the SLICE columns and run mma.sync m16n8k16 (bf16, fp32
// accumulation) on fragments read with ldmatrix from the swizzled tiles.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstddef>
#include <cstdint>

#include "common.cuh"

namespace tffn {
namespace decode {

constexpr int SLICE = 128;              // output columns per unit
constexpr int KC = 128;                 // K rows per unit
constexpr int MAX_ROWS = 64;            // rows handled by this path
constexpr int MAX_STAGES = 5;
constexpr int CONSUMER_WARPS = 4;       // 32 columns each
constexpr int NUM_THREADS = 32 * (1 + CONSUMER_WARPS);
constexpr int KC1 = 64;                 // K rows per stage of the gated window layer 1
constexpr int W_BOX_BYTES = KC * 64 * 2;                 // 16 KiB: KC rows x 64 cols
constexpr int W_STAGE_BYTES = 2 * W_BOX_BYTES;           // 32 KiB

// Geometry of the kernel instance for MT tiles of 16 rows (up to 64 rows):
// the A (X or H) box slot holds ROWS = 16 MT rows of 64 k; a stage is the W
// tile plus two A boxes; NST stages are in flight (measured on the 16-row
// instance: 4, 5 and the former 5 stages of 32-row slots stream alike at
// ~6.35 TB/s, 6 stages are 2 % slower, so it keeps 4 and leaves the rest of
// the shared memory to L1); KB k-steps of fragments are loaded before their
// MMAs (fewer for more rows: registers).
template <int MT>
struct Geo {
    static constexpr int ROWS = 16 * MT;
    static constexpr int A_BOX = ROWS * 64 * 2;
    static constexpr int STAGE = W_STAGE_BYTES + 2 * A_BOX;
    static constexpr int NST = MT == 1 ? 4 : (MT == 2 ? 5 : 4);
    static constexpr int SMEM = NST * STAGE + 1024 + 1024;
    static constexpr int KB = MT <= 2 ? 4 : 2;
};
static_assert(Geo<4>::SMEM <= 232448 && Geo<2>::SMEM <= 232448 && Geo<1>::SMEM <= 232448, "shared memory");
static_assert(Geo<1>::NST <= MAX_STAGES && Geo<2>::NST <= MAX_STAGES && Geo<4>::NST <= MAX_STAGES, "stages");

// Rows of a partial-sum block for M rows (the kernel instance's ROWS).
inline int decode_rows(int64_t M)
{
    return M <= 32 ? 32 : 64;
}

struct Plan {
    int32_t grid;
    // Gated window layer 1 (up to 32 rows): CTA c owns the 64-column hidden
    // blocks [c * nblk / grid, (c + 1) * nblk / grid) (one or two) and
    // computes the 128 columns of W1 and of W3 from its first block over all
    // of K in 64-row chunks (the second block of a one-block CTA is its
    // neighbour's, computed and dropped): no split slices in layer 1, H final
    // when the CTA's stream ends, one ready word per block and owning warp.
    int32_t win;
    int32_t nblk;
    int32_t h_per_k;        // layer-1 slices of H per layer-2 K chunk (1; 2 for the gated form)
    int32_t slices[2];      // output slices per layer
    int32_t kch[2];         // K chunks per slice
    int64_t units[2];       // slices * kch
    int32_t maxp[2];        // most CTAs sharing one slice
    int64_t part_off[2];    // float offset of each layer's partial area
    size_t partial_bytes;
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

// grid is the CTA count the caller wants; it is lowered so that every CTA
// owns at least one unit of each layer.
inline Plan make_plan(int64_t M, int64_t N, int64_t O, int64_t P, int grid, bool glu = false)
{
    Plan pl{};
    const int64_t rows = decode_rows(M);
    const int64_t h_cols = glu ? SLICE / 2 : SLICE;   // hidden columns per layer-1 slice
    pl.h_per_k = static_cast<int32_t>(KC / h_cols);
    pl.slices[0] = static_cast<int32_t>((O + h_cols - 1) / h_cols);
    pl.kch[0] = static_cast<int32_t>((N + KC - 1) / KC);
    pl.slices[1] = static_cast<int32_t>((P + SLICE - 1) / SLICE);
    pl.kch[1] = static_cast<int32_t>((O + KC - 1) / KC);
    int64_t g = grid;
    for (int l = 0; l < 2; ++l)
        pl.units[l] = static_cast<int64_t>(pl.slices[l]) * pl.kch[l];
    if (pl.units[1] < g)
        g = pl.units[1];
    if (g < 1)
        g = 1;
    pl.nblk = static_cast<int32_t>((O + 63) / 64);
    pl.win = (glu && M <= 32 && pl.nblk <= 2 * g) ? 1 : 0;
    if (pl.win) {
        pl.kch[0] = static_cast<int32_t>((N + KC1 - 1) / KC1);   // window chunks of KC1 rows
    } else if (pl.units[0] < g) {
        g = pl.units[0];
    }
    pl.grid = static_cast<int32_t>(g);
    size_t off = 0;
    for (int l = 0; l < 2; ++l) {
        if (l == 0 && pl.win) {
            pl.maxp[0] = 1;
            pl.part_off[0] = 0;
            continue;
        }
        int32_t maxp = 1;
        for (int64_t s = 0; s < pl.slices[l]; ++s) {
            const int64_t a = owner_of(s * pl.kch[l], pl.units[l], g);
            const int64_t b = owner_of((s + 1) * pl.kch[l] - 1, pl.units[l], g);
            if (b - a + 1 > maxp)
                maxp = static_cast<int32_t>(b - a + 1);
        }
        pl.maxp[l] = maxp;
        pl.part_off[l] = static_cast<int64_t>(off / 4);
        off += static_cast<size_t>(pl.slices[l]) * maxp * rows * SLICE * 4;
    }
    pl.partial_bytes = off;
    return pl;
}

struct Params {
    CUtensorMap map_w[2];      // W1 {O, N}, W2 {P, O}; box {64, KC} (gated window: W1 box {64, KC1})
    CUtensorMap map_a[2];      // X {N, M}, H {O, M}; box {64, 16 * m_tiles}
    CUtensorMap map_w3;        // gated form: W3 {O, N}; box {64, KC} (window: {64, KC1})
    const __nv_bfloat16* X;
    const __nv_bfloat16* W1;
    const __nv_bfloat16* b1;
    const __nv_bfloat16* W2;
    const __nv_bfloat16* b2;
    __nv_bfloat16* Y;
    __nv_bfloat16* H;          // [M x O]
    float* partial;
    uint32_t* counters;        // [slices0 * 4] then [slices1 * 4]
    uint32_t* flags;           // [slices0 * 4]: one word per consumer warp, = epoch when ready
                               // (gated window: [nblk * 2], one per block and owning warp)
    DevCtrl* ctrl;
    int32_t M, N, O, P;
    int32_t act1, act2;
    int32_t glu;               // 1: layer 1 is gated (no biases)
    int32_t skip_slice;        // test fault injection: this dense layer-1 slice's H flags are
                               // never published (-1 = off); its readers then time out
    uint64_t wait_limit_ns;
    Plan plan;
};

}  // namespace decode
}  // namespace tffn
