// noalloc.cu -- ffn_forward_decode_noalloc: the small-M (decode) FFN without
// any memory allocation, for callers that cannot allocate device memory.
//
// Its scratch (control word, ready flags, split-K counters, the hidden rows H
// and the split-K partial sums) lives in one file-scope __device__ array of
// NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds until
// the process exits.  The host never passes the array's name to a kernel: in
// host code that name is only a host-side stand-in, so the device address is
// fetched with cudaGetSymbolAddress once per device, with that device current.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/tffn.h"
#include "decode.cuh"
#include "launch.h"

static constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(16) << 20;   // 16 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

namespace {

struct NoallocDevice {
    bool ready = false;
    int sms = 0;
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
};

std::mutex g_noalloc_mu;
NoallocDevice g_noalloc_dev[64];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_noalloc_encode = nullptr;

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

int map2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer)
{
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_noalloc_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? 0
               : -1;
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim8(int64_t d) { return d >= 8 && d % 8 == 0 && d < (int64_t(1) << 31); }
bool act_valid(int a) { return a == TFFN_ACT_NONE || a == TFFN_ACT_RELU || a == TFFN_ACT_GELU_TANH || a == TFFN_ACT_SILU; }

// One-time set-up of the current device: the array's device address, the SM
// count and the tensor-map encoder.
int noalloc_setup(NoallocDevice** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return TFFN_ERR_CUDA;
    NoallocDevice& d = g_noalloc_dev[dev];
    if (!d.ready) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return TFFN_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TFFN_ERR_CUDA;
        if (!g_noalloc_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return TFFN_ERR_CUDA;
            g_noalloc_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.scratch = static_cast<unsigned char*>(ptr);
        d.ready = true;
    }
    *out = &d;
    return TFFN_OK;
}

}  // namespace

extern "C" int ffn_forward_decode_noalloc(const void* X, const void* W1, const void* b1, const void* W2,
                                          const void* b2, int act1, int act2, int64_t M, int64_t N, int64_t O,
                                          int64_t P, void* Y, struct CUstream_st* stream)
{
    using namespace tffn;
    if (M < 0 || M > 32 || !dim8(N) || !dim8(O) || !dim8(P) || !act_valid(act1) ||
        !act_valid(act2))
        return TFFN_ERR_INVALID_ARG;
    if (M == 0)
        return TFFN_OK;
    if (!X || !W1 || !W2 || !Y || !a16(X) || !a16(W1) || !a16(W2) || !a16(Y) || (b1 && !a16(b1)) ||
        (b2 && !a16(b2)))
        return TFFN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocDevice* d = nullptr;
    int rc = noalloc_setup(&d);
    if (rc != TFFN_OK)
        return rc;

    decode::Params p{};
    p.plan = decode::make_plan(M, N, O, P, d->sms);
    // Scratch layout: control block | flags | counters | H | partial sums.
    const size_t off_flags = 256;
    const size_t flag_words = static_cast<size_t>(p.plan.slices[0]) * decode::CONSUMER_WARPS;
    const size_t off_counters = up256(off_flags + flag_words * 4);
    const size_t counter_words =
        (static_cast<size_t>(p.plan.slices[0]) + p.plan.slices[1]) * decode::CONSUMER_WARPS;
    const size_t zeroed = up256(off_counters + counter_words * 4);
    const size_t off_h = zeroed;
    const size_t off_part = up256(off_h + static_cast<size_t>(M) * O * 2);
    const size_t need = off_part + p.plan.partial_bytes;
    if (need > NOALLOC_SCRATCH_BYTES)
        return TFFN_ERR_UNSUPPORTED;   // shape needs more scratch than the static array holds

    unsigned char* base = d->scratch;
    // Control word, flags and counters start every call at zero (the array
    // keeps whatever the previous call left there).
    if (cudaMemsetAsync(base, 0, zeroed, s) != cudaSuccess)
        return TFFN_ERR_CUDA;
    p.X = static_cast<const __nv_bfloat16*>(X);
    p.W1 = static_cast<const __nv_bfloat16*>(W1);
    p.b1 = static_cast<const __nv_bfloat16*>(b1);
    p.W2 = static_cast<const __nv_bfloat16*>(W2);
    p.b2 = static_cast<const __nv_bfloat16*>(b2);
    p.Y = static_cast<__nv_bfloat16*>(Y);
    p.H = reinterpret_cast<__nv_bfloat16*>(base + off_h);
    p.partial = reinterpret_cast<float*>(base + off_part);
    p.counters = reinterpret_cast<uint32_t*>(base + off_counters);
    p.flags = reinterpret_cast<uint32_t*>(base + off_flags);
    p.ctrl = reinterpret_cast<DevCtrl*>(base);
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.O = static_cast<int32_t>(O);
    p.P = static_cast<int32_t>(P);
    p.act1 = act1;
    p.act2 = act2;   // flags and epoch were just cleared: the kernel uses epoch 1
    p.skip_slice = option_skip_flag();
    p.wait_limit_ns = option_wait_limit_ns();
    const uint32_t arows = M <= 16 ? 16u : 32u;
    if (map2d(&p.map_w[0], W1, O, N, 64, decode::KC) || map2d(&p.map_w[1], W2, P, O, 64, decode::KC) ||
        map2d(&p.map_a[0], X, N, M, 64, arows) || map2d(&p.map_a[1], p.H, O, M, 64, arows))
        return TFFN_ERR_INVALID_ARG;
    if (launch_decode(p, p.plan.grid, s) != 0)
        return TFFN_ERR_CUDA;
    return TFFN_OK;
}

extern "C" int tffn_check_noalloc(struct CUstream_st* stream, int32_t* detail)
{
    if (detail)
        detail[0] = detail[1] = detail[2] = detail[3] = 0;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TFFN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return TFFN_ERR_CUDA;
    const NoallocDevice& d = g_noalloc_dev[dev];
    if (!d.ready)
        return TFFN_OK;   // no call has run on this device
    // The first four words of the control block: {status, wait site, block, info}.
    uint32_t rec[4] = {0, 0, 0, 0};
    if (cudaMemcpy(rec, d.scratch, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TFFN_ERR_CUDA;
    if (detail)
        for (int i = 0; i < 4; ++i)
            detail[i] = static_cast<int32_t>(rec[i]);
    if (rec[0] == 0)
        return TFFN_OK;
    if (cudaMemset(d.scratch, 0, sizeof(rec)) != cudaSuccess)
        return TFFN_ERR_CUDA;
    return static_cast<int32_t>(rec[0]) == TFFN_ERR_TIMEOUT ? TFFN_ERR_TIMEOUT : TFFN_ERR_DEVICE;
}
