// engine_grouped.cu -- the engine instantiated for up to 64 experts
// (moe_ffn_forward): each row band belongs to one expert and selects that
// expert's weight maps and biases.
#include "engine_launch.cuh"
#include "launch.h"

namespace tffn {

// Kernel parameters are limited to 32764 bytes.
static_assert(sizeof(engine::Params<MOE_MAX_E>) <= 32764, "grouped engine parameters fit a launch");

int launch_engine_grouped(const engine::Params<MOE_MAX_E>& p, int max_pairs, cudaStream_t s)
{
    return launch_engine_pairs<MOE_MAX_E>(p, max_pairs, s);
}

}  // namespace tffn
