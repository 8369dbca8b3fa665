// common.cuh -- device-side control block, error reporting and bounded waits.
//
// Every wait in the library's kernels goes through wait_mbar / wait_flag: each
// has a time limit (globaltimer, nanoseconds) after which the kernel records an
// error in the workspace's control block, raises the CTA's abort flag and
// returns, so the host can read the error from tffn_check() and the context
// stays usable.  Nothing traps.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "../../include/tffn.h"
#include "ptx.cuh"

namespace tffn {

// Where a wait gave up (stored in DevCtrl::where).
enum WaitSite : uint32_t {
    SITE_SMEM_EMPTY = 1,     // producer waiting for a free shared-memory stage
    SITE_SMEM_FULL = 2,      // MMA waiting for a loaded stage
    SITE_TMEM_EMPTY = 3,     // MMA waiting for a drained accumulator
    SITE_TMEM_FULL = 4,      // epilogue waiting for a finished accumulator
    SITE_TASK_FULL = 5,      // consumer waiting for the next task
    SITE_TASK_EMPTY = 6,     // producer waiting for a free task slot
    SITE_H_FLAG = 7,         // layer-2 producer waiting for a hidden tile
    SITE_DRAIN = 8,          // exit path waiting for its own copies / MMAs
    SITE_SLICE_FLAG = 9,     // decode layer 2 waiting for a hidden slice
    SITE_STAGE = 10,         // decode consumer waiting for a stage
    SITE_H_SMEM = 11,        // reduce-add form: MMA waiting for the H tile in shared memory
    SITE_H_FREE = 12,        // reduce-add form: epilogue waiting for the H tile's readers
    SITE_BIAS = 13,          // engine epilogue: the CTA's shared bias slice
    SITE_PARTS = 14,         // weight streams: a slice's reducer waiting for its split-K parts
};

// Control block at the start of the workspace (256 bytes).
struct DevCtrl {
    uint32_t status;      // 0 or a negative tffn_status, stored as uint32
    uint32_t where;       // WaitSite of the first failure
    uint32_t block;       // blockIdx.x of the first failure
    uint32_t info;        // site-specific detail (tile / slice index)
    uint32_t ticket;      // engine: next task ticket
    uint32_t done;        // engine: CTAs that have exited
    uint32_t epoch;       // ready-flag value of the most recent launch; each launch
                          // stamps and expects epoch + 1 and the last CTA out stores it
    uint32_t ddone;       // decode: CTAs that have exited
    uint32_t pad[56];
};
static_assert(sizeof(DevCtrl) == 256, "control block is 256 bytes");

struct WaitCtx {
    volatile uint32_t* abort;   // CTA-wide abort flag in shared memory
    DevCtrl* ctrl;
    uint64_t limit_ns;
    uint32_t peer_abort;        // shared::cluster address of the peer CTA's abort flag (0: none)
};

__device__ __forceinline__ void raise_error(const WaitCtx& w, uint32_t code, uint32_t where,
                                            uint32_t info)
{
    *w.abort = 1u;
    if (w.peer_abort != 0u)
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(w.peer_abort), "r"(1u) : "memory");
    if (atomicCAS(&w.ctrl->status, 0u, code) == 0u) {
        w.ctrl->where = where;
        w.ctrl->block = blockIdx.x;
        w.ctrl->info = info;
    }
}

// Polls made inline before a wait falls back to its timed loop.  The hot
// loops (a stage ring's full / empty barriers) wait on every k-block; an
// out-of-line call there cost the engine 4-8 % (GEMM of 4096 x 4096 x 16384:
// 357 -> 328 us with the inline polls).
constexpr int FAST_POLLS = 4096;

// The timed part of wait_mbar (out of line: rarely reached).
static __device__ __noinline__ bool wait_mbar_timed(const WaitCtx& w, uint32_t bar, uint32_t parity,
                                                    uint32_t where)
{
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if (*w.abort)
            return false;
        if (ptx::globaltimer() - t0 > w.limit_ns) {
            raise_error(w, static_cast<uint32_t>(TFFN_ERR_TIMEOUT), where, parity);
            return false;
        }
    }
}

// Wait for the phase of `bar` with this parity: at most FAST_POLLS inline
// probes, then the timed loop; false on abort or timeout.
__device__ __forceinline__ bool wait_mbar(const WaitCtx& w, uint32_t bar, uint32_t parity, uint32_t where)
{
#pragma unroll 1
    for (int i = 0; i < FAST_POLLS; ++i)
        if (ptx::mbar_try_wait(bar, parity))
            return true;
    return wait_mbar_timed(w, bar, parity, where);
}

// The timed part of wait_mbar_cl.
static __device__ __noinline__ bool wait_mbar_cl_timed(const WaitCtx& w, uint32_t bar, uint32_t parity,
                                                       uint32_t where)
{
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait_cluster(bar, parity))
            return true;
        if (*w.abort)
            return false;
        if (ptx::globaltimer() - t0 > w.limit_ns) {
            raise_error(w, static_cast<uint32_t>(TFFN_ERR_TIMEOUT), where, parity);
            return false;
        }
    }
}

// Same, acquiring at cluster scope: for barriers that receive arrivals from the
// peer CTA of a cluster (or from its tensor-core commits).
__device__ __forceinline__ bool wait_mbar_cl(const WaitCtx& w, uint32_t bar, uint32_t parity, uint32_t where)
{
#pragma unroll 1
    for (int i = 0; i < FAST_POLLS; ++i)
        if (ptx::mbar_try_wait_cluster(bar, parity))
            return true;
    return wait_mbar_cl_timed(w, bar, parity, where);
}

// Wait (acquire, gpu scope) until *flag == epoch; false on abort or timeout.
static __device__ __noinline__ bool wait_flag(const WaitCtx& w, const uint32_t* flag, uint32_t epoch,
                                       uint32_t where, uint32_t info)
{
    if (ptx::ld_acquire_gpu(flag) == epoch)
        return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        __nanosleep(100);
        if (ptx::ld_acquire_gpu(flag) == epoch)
            return true;
        if (*w.abort)
            return false;
        if (ptx::globaltimer() - t0 > w.limit_ns) {
            raise_error(w, static_cast<uint32_t>(TFFN_ERR_TIMEOUT), where, info);
            return false;
        }
    }
}

// Activations (fp32).  GELU uses the tanh form written through the identity
// 0.5 x (1 + tanh(u)) = x / (1 + exp(-2u)), which keeps full relative accuracy
// for negative x where 1 + tanh(u) would cancel.  With u = sqrt(2/pi) (x +
// 0.044715 x^3), exp(-2u) = 2^(x (c0 + c1 x^2)) for c0 = -2 sqrt(2/pi) log2(e)
// and c1 = 0.044715 c0: three multiply-adds before the base-2 exponential
// (the epilogue's activation arithmetic shows in the whole launch's time).
// A very negative x gives 2^y = inf and a result of -0, GELU's limit; below
// 2^-126 (x beyond ~10) the exponential flushes to 0 and the result is x.
// SiLU is x sigma(x) = x / (1 + exp(-x)), exp(-x) taken the same way; the
// exponent is capped at 80 so the denominator stays finite (below x = -80
// the result is below 1e-33 in magnitude either way).
__device__ __forceinline__ float ex2_approx(float y)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

__device__ __forceinline__ float act_apply(int act, float x)
{
    if (act == TFFN_ACT_RELU)
        return fmaxf(x, 0.0f);
    if (act == TFFN_ACT_GELU_TANH) {
        const float c0 = -2.3022082f;    // -2 sqrt(2/pi) / ln 2
        const float c1 = -0.10294324f;   // 0.044715 c0
        const float e = ex2_approx(x * fmaf(c1, x * x, c0));
        return __fdividef(x, 1.0f + e);
    }
    if (act == TFFN_ACT_SILU)
        return __fdividef(x, 1.0f + ex2_approx(fmaxf(x, -80.0f) * -1.44269504f));   // exp(-x) = 2^(-x / ln 2)
    return x;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v)
{
    return __uint_as_float(v << 16);
}

__device__ __forceinline__ float bf16_hi(uint32_t v)
{
    return __uint_as_float(v & 0xFFFF0000u);
}

}  // namespace tffn
