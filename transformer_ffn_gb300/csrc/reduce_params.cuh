// reduce_params.cuh -- constants, launch parameters and shared-memory block
// of the reduce-add form of the fused FFN (kernel in reduce.cuh).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "engine.cuh"

namespace tffn {
namespace reduce {

using engine::A_STAGE_BYTES;
using engine::B_BOX_BYTES;
using engine::B_LOADER_WARP;
using engine::B_STAGE_BYTES;
using engine::BK;
using engine::BM;
using engine::BM_CTA;
using engine::BN;
using engine::BN_CTA;
using engine::EPI_WARPS;
using engine::NUM_THREADS;
using engine::STAGE_BYTES;
using engine::TASK_CONSUMERS;
using engine::TASK_SLOTS;
using engine::TMEM_COLS;

constexpr int STAGES = 4;
constexpr int H_BLOCK_BYTES = BM_CTA * 64 * 2;            // 128 rows x 64 hidden columns, bf16
constexpr int H_BYTES = (BN / 64) * H_BLOCK_BYTES;         // 64 KiB
constexpr int STG_BYTES = 32 * 32 * 4;                     // one warp's 32 rows x 32 fp32 columns
constexpr int STG_BUFS = 2;
constexpr int AUX_BYTES = 1024;
constexpr int OFF_H = STAGES * STAGE_BYTES;
constexpr int OFF_STG = OFF_H + H_BYTES;
constexpr int OFF_AUX = OFF_STG + EPI_WARPS * STG_BUFS * STG_BYTES;
constexpr int SMEM_BYTES = OFF_AUX + AUX_BYTES + 1024;     // + alignment slack
constexpr int COUNTERS_PER_TILE = 2 * EPI_WARPS;           // one per 32-row strip of a Y tile
constexpr int CHUNKS = BN / 32;                            // 32-column chunks of a tile

struct Params {
    CUtensorMap map_x;      // X [M x N] bf16, box {64, 128}
    CUtensorMap map_w1;     // W1 [N x O] bf16, as the engine's B maps
    CUtensorMap map_w2;     // W2 [O x P] bf16, as the engine's B maps
    CUtensorMap map_acc;    // Y accumulator [m_blocks*256 x P] fp32, box {32, 32}, 128-byte swizzle
    const __nv_bfloat16* b1;   // nullable
    const __nv_bfloat16* b2;   // nullable
    const float* acc;          // the Y accumulator, read back by the last contributor
    __nv_bfloat16* Y;          // [M x P]
    uint32_t* counters;        // [m_blocks * n_p * COUNTERS_PER_TILE], zero at launch
    DevCtrl* ctrl;
    uint64_t wait_limit_ns;
    int64_t M;
    int32_t N, O, P;
    int32_t act1, act2;
    int32_t m_blocks, n_h, n_p;   // bands, hidden tiles, Y column tiles
    int32_t b3d;
};

struct Aux {
    uint64_t full[STAGES];          // leader: the TMA bytes of both CTAs
    uint64_t empty[STAGES];         // MMA done with the stage (multicast commit)
    uint64_t tmem_full[2];          // accumulator ready (multicast commit)
    uint64_t tmem_empty[2];         // leader: the pair's eight epilogue warps drained it
    uint64_t h_full;                // leader: the pair's eight epilogue warps wrote the H tile
    uint64_t h_empty;               // the MMAs reading the H tile are done (multicast commit)
    uint64_t task_full[TASK_SLOTS];
    uint64_t task_empty[TASK_SLOTS];
    uint64_t drain;
    int4 task[TASK_SLOTS];
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(Aux) <= AUX_BYTES, "aux block fits");
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

}  // namespace reduce
}  // namespace tffn
