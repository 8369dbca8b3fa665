// engine_grouped.cu -- the engine instantiated for up to 64 experts
// (moe_ffn_forward): each row band belongs to one expert and selects that
// expert's weight maps and biases.
#include "engine_launch.cuh"
#include "launch.h"

namespace tffn {

int launch_engine_grouped(const engine::Params<MOE_MAX_E>& p, int max_pairs, cudaStream_t s)
{
    return launch_engine_pairs<MOE_MAX_E>(p, max_pairs, s);
}

}  // namespace tffn
