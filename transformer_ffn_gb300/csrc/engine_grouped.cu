// engine_grouped.cu -- the engine instantiated for up to 64 experts
// (moe_ffn_forward): each row band belongs to one expert and selects that
// expert's weight maps and biases.
#include "engine.cuh"
#include "launch.h"

namespace tffn {

int launch_engine_grouped(const engine::Params<MOE_MAX_E>& p, int grid, cudaStream_t s)
{
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(engine::engine_kernel<MOE_MAX_E>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, engine::SMEM_BYTES) != cudaSuccess)
            return -1;
        attr_set = true;
    }
    engine::engine_kernel<MOE_MAX_E><<<grid, engine::NUM_THREADS, engine::SMEM_BYTES, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tffn
