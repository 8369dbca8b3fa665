// engine_dense.cu -- the engine instantiated for one weight set (ffn_forward).
#include "engine.cuh"
#include "launch.h"

namespace tffn {

int launch_engine_dense(const engine::Params<1>& p, int grid, cudaStream_t s)
{
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(engine::engine_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 engine::SMEM_BYTES) != cudaSuccess)
            return -1;
        attr_set = true;
    }
    engine::engine_kernel<1><<<grid, engine::NUM_THREADS, engine::SMEM_BYTES, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tffn
