// engine_launch.cuh -- cluster launch of the 2-SM engine (clusters of two
// CTAs), with the grid capped at the number of CTA pairs the GPU can keep
// resident at once (the engine is persistent: every CTA stays until the
// ticket queue is empty).
#pragma once

#include <cuda_runtime.h>

#include "engine.cuh"

namespace tffn {

template <int MAX_E>
int launch_engine_pairs(const engine::Params<MAX_E>& p, int max_pairs, cudaStream_t s)
{
    static bool ready = false;
    static int resident_pairs = 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(engine::NUM_THREADS);
    cfg.dynamicSmemBytes = engine::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!ready) {
        if (cudaFuncSetAttribute(engine::engine_kernel<MAX_E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 engine::SMEM_BYTES) != cudaSuccess)
            return -1;
        cfg.gridDim = dim3(2);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, engine::engine_kernel<MAX_E>, &cfg) != cudaSuccess || n < 1)
            return -1;
        resident_pairs = n;
        ready = true;
    }
    int pairs = max_pairs < resident_pairs ? max_pairs : resident_pairs;
    if (pairs < 1)
        pairs = 1;
    cfg.gridDim = dim3(2 * pairs);
    if (cudaLaunchKernelEx(&cfg, engine::engine_kernel<MAX_E>, p) != cudaSuccess)
        return -1;
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tffn
