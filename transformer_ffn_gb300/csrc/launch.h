// launch.h -- host-side launchers of the library's kernels (one per
// translation unit), called by api.cu.  Every launcher returns 0 or -1 (launch
// error; the CUDA error is left for the caller to read).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tffn {
namespace engine {
template <int MAX_E>
struct Params;
}
namespace decode {
struct Params;
}
namespace reduce {
struct Params;
}
namespace wstream {
struct Params;
}

constexpr int MOE_MAX_E = 64;

// Process-wide options shared by every entry point (tffn_set_option):
// the device wait limit in nanoseconds and the test fault-injection index
// (-1 = off).
uint64_t option_wait_limit_ns();
int32_t option_skip_flag();

// The engine launches clusters of two CTAs; max_pairs caps the number of CTA
// pairs (further capped by how many pairs can be resident at once).
int launch_engine_dense(const engine::Params<1>& p, int max_pairs, cudaStream_t s);
int launch_engine_grouped(const engine::Params<MOE_MAX_E>& p, int max_pairs, cudaStream_t s);
int launch_decode(const decode::Params& p, int grid, cudaStream_t s);
int launch_wstream(const wstream::Params& p, cudaStream_t s);
int launch_reduce(const reduce::Params& p, int max_pairs, cudaStream_t s);
int launch_b2b(const reduce::Params& p, int max_pairs, cudaStream_t s);

// Token blocks of the MoE routing (per-block expert counts, per-block scatter).
int moe_route_blocks(int64_t T);
int launch_moe_route(const float* logits, int64_t T, int E, int k, int32_t* idx, float* w, int32_t* blk_hist,
                     cudaStream_t s);
int launch_moe_plan(const int32_t* blk_hist, int64_t T, int E, int bm, int size_desc, int32_t* blk_pad,
                    int32_t* blk_off, int32_t* band_expert, int32_t* nbands, int32_t* pad, int32_t* offs_out,
                    cudaStream_t s);
// row_entry (nullable): the routing entry of each grouped row, -1 for padding rows
// (the scatter writes the real rows, the gather the padding rows).
int launch_moe_scatter(const int32_t* idx, int64_t T, int E, int k, const int32_t* blk_pad, const int32_t* blk_off,
                       int32_t* pos, int32_t* perm_out, int32_t* row_entry, cudaStream_t s);
int launch_moe_gather(const void* X, const int32_t* pos, int64_t T, int k, const int32_t* pad, int E, int64_t N,
                      void* Xp, int32_t* row_entry, int grid, cudaStream_t s);
int launch_moe_combine(const float* Yp, const int32_t* pos, const float* w, int64_t T, int k, int64_t P,
                       void* Y, int grid, cudaStream_t s);

}  // namespace tffn
