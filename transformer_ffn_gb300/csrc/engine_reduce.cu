// engine_reduce.cu -- cluster launches of the reduce-add and back-to-back
// forms (reduce.cuh): clusters of two CTAs, grid capped at the CTA pairs the
// GPU keeps resident.
#include <cuda_runtime.h>

#include "launch.h"
#include "reduce.cuh"

namespace tffn {

namespace {

using KernelFn = void (*)(reduce::Params);

int launch_pairs(KernelFn kernel, bool& ready, int& resident_pairs, const reduce::Params& p, int max_pairs,
                 cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(reduce::NUM_THREADS);
    cfg.dynamicSmemBytes = reduce::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!ready) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, reduce::SMEM_BYTES) !=
            cudaSuccess)
            return -1;
        cfg.gridDim = dim3(2);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1)
            return -1;
        resident_pairs = n;
        ready = true;
    }
    int pairs = max_pairs < resident_pairs ? max_pairs : resident_pairs;
    if (pairs < 1)
        pairs = 1;
    cfg.gridDim = dim3(2 * pairs);
    if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess)
        return -1;
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_reduce(const reduce::Params& p, int max_pairs, cudaStream_t s)
{
    static bool ready = false;
    static int resident_pairs = 0;
    return launch_pairs(reduce::reduce_kernel, ready, resident_pairs, p, max_pairs, s);
}

int launch_b2b(const reduce::Params& p, int max_pairs, cudaStream_t s)
{
    static bool ready = false;
    static int resident_pairs = 0;
    return launch_pairs(reduce::b2b_kernel, ready, resident_pairs, p, max_pairs, s);
}

}  // namespace tffn
