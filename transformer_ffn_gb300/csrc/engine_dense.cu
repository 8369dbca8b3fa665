// engine_dense.cu -- the engine instantiated for one weight set (ffn_forward).
#include "engine_launch.cuh"
#include "launch.h"

namespace tffn {

int launch_engine_dense(const engine::Params<1>& p, int max_pairs, cudaStream_t s)
{
    return launch_engine_pairs<1>(p, max_pairs, s);
}

}  // namespace tffn
