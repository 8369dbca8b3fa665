// schedule.h -- the engine's task order, shared by the kernel and the host.
//
// One fused launch runs two kinds of output tiles: layer-1 tiles (a band of BM
// rows of H times BN columns) and layer-2 tiles (a band of BM rows of Y times
// BN columns).  A layer-2 tile of band i reads the whole H band i, so it waits
// on the ready flags of every layer-1 tile of that band ("Kernel fusion and
// tensor parallelism", section "Step 1": a tile of H feeds the row of Y tiles
// as soon as it is ready; the per-tile flag of the same section).
//
// Tickets are handed out in increasing order by an atomic counter.  Bands are
// taken in raster groups of `group_m` bands; inside a group, tiles go column
// tile by column tile, so concurrently running tiles share weight panels in L2.
// The sequence of segments is
//     L1(g0), L1(g1), L2(g0), L1(g2), L2(g1), ..., L1(g_last), L2(g_prev), L2(g_last)
// so every layer-2 tile comes after all layer-1 tiles it depends on, one group
// later: a task only ever waits on tasks with smaller tickets, which makes the
// persistent launch deadlock-free for any number of resident CTAs >= 1.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define TFFN_HD __host__ __device__ __forceinline__
#else
#define TFFN_HD inline
#endif

namespace tffn {

struct EngineTask {
    int32_t layer;   // 0 = layer 1 (H), 1 = layer 2 (Y), -1 = no more work
    int32_t band;    // row band (BM rows)
    int32_t tile;    // column tile (BN columns)
};

enum EngineMode : int32_t {
    MODE_FUSED = 0,     // both layers, layer 2 waits on layer-1 flags
    MODE_LAYER1 = 1,    // layer 1 only
    MODE_LAYER2 = 2     // layer 2 only (H already complete)
};

TFFN_HD int64_t engine_total_tickets(int64_t m_blocks, int32_t n1, int32_t n2, int32_t mode)
{
    if (mode == MODE_LAYER1)
        return m_blocks * n1;
    if (mode == MODE_LAYER2)
        return m_blocks * n2;
    return m_blocks * (static_cast<int64_t>(n1) + n2);
}

// The mapping is written once for any signed index type I: the host and the
// schedule tests use int64_t; the kernel uses int32_t (32-bit division is
// several times cheaper than 64-bit division on the GPU, and the host refuses
// launches whose ticket count does not fit in 31 bits).
template <typename I>
TFFN_HD EngineTask engine_in_group_t(int32_t layer, I group, I idx, I m_blocks, I group_m)
{
    const I first = group * group_m;
    const I gsize = m_blocks - first < group_m ? m_blocks - first : group_m;
    EngineTask r;
    r.layer = layer;
    r.band = static_cast<int32_t>(first + idx % gsize);
    r.tile = static_cast<int32_t>(idx / gsize);
    return r;
}

template <typename I>
TFFN_HD EngineTask engine_task_t(I t, I m_blocks, I n1, I n2, I group_m, int32_t mode)
{
    EngineTask end;
    end.layer = -1;
    end.band = 0;
    end.tile = 0;
    if (t < 0 || m_blocks <= 0)
        return end;
    const I ng = (m_blocks + group_m - 1) / group_m;

    if (mode == MODE_LAYER1 || mode == MODE_LAYER2) {
        const I n = mode == MODE_LAYER1 ? n1 : n2;
        if (t >= m_blocks * n)
            return end;
        const I g = t / (group_m * n);
        return engine_in_group_t<I>(mode == MODE_LAYER1 ? 0 : 1, g, t - g * group_m * n, m_blocks, group_m);
    }

    auto gsize = [&](I g) -> I {
        const I rest = m_blocks - g * group_m;
        return rest < group_m ? rest : group_m;
    };
    // L1(g0)
    I len = gsize(0) * n1;
    if (t < len)
        return engine_in_group_t<I>(0, 0, t, m_blocks, group_m);
    t -= len;
    // pairs [L1(g), L2(g-1)] for g = 1 .. ng-1; pairs 1 .. ng-2 are full-sized
    // (only the last group can be short), so whole pairs are skipped at once
    I g0 = 1;
    if (ng >= 3) {
        const I pair = group_m * (n1 + n2);
        I skip = t / pair;
        if (skip > ng - 2)
            skip = ng - 2;
        t -= skip * pair;
        g0 += skip;
    }
    for (I g = g0; g < ng; ++g) {
        len = gsize(g) * n1;
        if (t < len)
            return engine_in_group_t<I>(0, g, t, m_blocks, group_m);
        t -= len;
        len = gsize(g - 1) * n2;
        if (t < len)
            return engine_in_group_t<I>(1, g - 1, t, m_blocks, group_m);
        t -= len;
    }
    // L2(g_last)
    len = gsize(ng - 1) * n2;
    if (t < len)
        return engine_in_group_t<I>(1, ng - 1, t, m_blocks, group_m);
    return end;
}

TFFN_HD EngineTask engine_task(int64_t t, int64_t m_blocks, int32_t n1, int32_t n2, int32_t group_m,
                               int32_t mode)
{
    return engine_task_t<int64_t>(t, m_blocks, n1, n2, group_m, mode);
}

// Largest ticket count a launch may have: the kernel's ticket counter and its
// task arithmetic are 32-bit, and every pair takes one ticket past the end.
constexpr int64_t ENGINE_MAX_TICKETS = (int64_t(1) << 31) - (int64_t(1) << 16);

}  // namespace tffn
