// api.cu -- the C ABI (include/tffn.h): argument validation, the workspace,
// tensor-map encoding and kernel launches.  No arithmetic of the FFN happens
// here; every step of the path runs in the kernels of this directory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <memory>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/tffn.h"
#include "decode.cuh"
#include "wstream.cuh"
#include "engine.cuh"
#include "launch.h"
#include "reduce_params.cuh"
#include "schedule.h"

namespace {

using namespace tffn;

// ----------------------------------------------------------- workspace map
// [0, 256)                 DevCtrl
// [256, 256 + 4 MiB)       ready flags / counters (engine: one per layer-1 tile)
// [.., + 256 KiB)          decode split-K arrival counters
// [.., + 64 KiB)           engine band counts
// [.., SYNC_BYTES)         MoE combine arrival counters
// [SYNC_BYTES, ...)        data: H, grouped rows, partial sums
// The sync region is zeroed when a workspace is (re)initialised; after that,
// flags are compared against the epoch kept in the control block (advanced by
// every launch on the device, so CUDA-graph replays stay correct) and counters
// are reset by the kernels: no per-call clearing is needed.
constexpr size_t OFF_FLAGS = 256;
constexpr size_t FLAG_WORDS = size_t(1) << 20;
constexpr size_t OFF_DCOUNT = OFF_FLAGS + FLAG_WORDS * 4;
constexpr size_t DCOUNT_WORDS = size_t(1) << 16;
constexpr size_t SYNC_BYTES = size_t(5) << 20;
// Engine band counts (two per 256-row band), zeroed by the last CTA out of
// every fused engine launch; used by nothing else.
constexpr size_t OFF_BCOUNT = OFF_DCOUNT + DCOUNT_WORDS * 4;
constexpr size_t BCOUNT_WORDS = size_t(1) << 14;
// MoE combine arrival counters (one per token and Y column tile), reset by
// the last arriver, in the rest of the sync region.
constexpr size_t OFF_MCOUNT = OFF_BCOUNT + BCOUNT_WORDS * 4;
constexpr size_t MCOUNT_WORDS = (SYNC_BYTES - OFF_MCOUNT) / 4;
static_assert(OFF_MCOUNT < SYNC_BYTES, "sync region layout");
constexpr uint32_t EPOCH_LIMIT = 0x7FFFFFF0u;      // launches before the flag region is cleared

// The band counts of a fused engine launch over `bands` bands (NULL when
// there are more bands than the region holds: the producers then poll the
// per-tile flags only).
static uint32_t* band_counts(uint8_t* base, int64_t bands)
{
    return static_cast<size_t>(bands) * 2 <= BCOUNT_WORDS ? reinterpret_cast<uint32_t*>(base + OFF_BCOUNT) : nullptr;
}

constexpr int64_t DECODE_MAX_M = 32;   // the mma.sync weight stream wins up to here (measured)
constexpr int64_t STREAM_MAX_M = 128;  // then the tensor-core weight stream, then the engine (measured);
                                       // up to 256 rows while its window layer 1 applies

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------ launch-parameter cache
// A forward call's kernel parameters -- the encoded tensor maps (a driver call
// each, a few microseconds together) and the work plan -- depend only on the
// call's pointers, shapes, activations, resolved path and workspace base.  The
// last few distinct calls per kind and device are kept; a repeated call (the
// same layer in a serving loop) launches from the cached copy after
// refreshing the fields that follow the process-wide options.  Tensor maps
// hold addresses and shapes only, so a cached entry stays valid whatever the
// tensors contain.
struct CallKey {
    int32_t kind = 0, path = 0, act1 = 0, act2 = 0;
    int64_t dims[6] = {0, 0, 0, 0, 0, 0};
    std::vector<const void*> ptrs;
    bool operator==(const CallKey& o) const
    {
        return kind == o.kind && path == o.path && act1 == o.act1 && act2 == o.act2 &&
               std::memcmp(dims, o.dims, sizeof(dims)) == 0 && ptrs == o.ptrs;
    }
};

template <class P>
struct ParamCache {
    static constexpr int SLOTS = 4;
    CallKey key[SLOTS];
    std::unique_ptr<P> params[SLOTS];
    int next = 0;
    P* find(const CallKey& k)
    {
        for (int i = 0; i < SLOTS; ++i)
            if (params[i] && key[i] == k)
                return params[i].get();
        return nullptr;
    }
    P* store(const CallKey& k, const P& p)
    {
        const int i = next;
        next = (next + 1) % SLOTS;
        key[i] = k;
        if (!params[i])
            params[i].reset(new P);
        std::memcpy(static_cast<void*>(params[i].get()), &p, sizeof(P));
        return params[i].get();
    }
};

struct DeviceState {
    bool init = false;
    int sms = 0;
    void* owned = nullptr;
    size_t owned_bytes = 0;
    void* user = nullptr;
    size_t user_bytes = 0;
    bool user_set = false;
    bool needs_reset = true;
    uint32_t launches = 0;   // flag-using launches since the flag region was cleared
    ParamCache<decode::Params> decode_cache;
    ParamCache<wstream::Params> wstream_cache;
    ParamCache<engine::Params<1>> engine_cache;
    ParamCache<engine::Params<MOE_MAX_E>> moe_cache;
};

std::mutex g_mu;
DeviceState g_dev[64];

std::atomic<int64_t> g_opt_path{0};
std::atomic<int64_t> g_opt_wait_ms{4000};
std::atomic<int64_t> g_opt_skip{-1};
std::atomic<int64_t> g_opt_group{0};
std::atomic<int64_t> g_opt_moe_order{1};
std::atomic<int64_t> g_opt_moe_combine{1};

thread_local int g_last_launches = 0;
thread_local bool g_timing = false;
thread_local int g_timing_every = 1;        // time one dominant launch of every g_timing_every
thread_local uint64_t g_timing_seen = 0;
thread_local bool g_timing_this = false;
thread_local std::vector<std::pair<cudaEvent_t, cudaEvent_t>> g_events;
thread_local size_t g_events_used = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int get_encode()
{
    if (g_encode)
        return 0;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return -1;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return 0;
}

// Row-major bf16 matrix [outer x inner], box [box_outer x box_inner], 128-byte
// swizzle, zero fill outside the matrix.
// promo: L2 sector promotion of each fetch (256 B by default; 128 B for
// boxes whose 128-byte rows are not followed by the same CTA's next box).
int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
             uint32_t box_outer, CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
{
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -1;
}

// W [K x ncols] row-major bf16 seen as {64 columns, K rows, ncols/64 column
// blocks}, box {64, 64, 2}: one copy brings a 64-deep, 128-column slab in the
// same shared-memory layout as two 2-D {64, 64} boxes.  Only for ncols % 64 == 0
// (a partial last block would reach past the end of the matrix).
int make_map_b3(CUtensorMap* m, const void* base, uint64_t ncols, uint64_t K)
{
    cuuint64_t dims[3] = {64, K, ncols / 64};
    cuuint64_t strides[2] = {ncols * 2, 128};
    cuuint32_t box[3] = {64, 64, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -1;
}

int make_map_b(CUtensorMap* m, const void* base, int64_t ncols, int64_t K, bool b3d)
{
    return b3d ? make_map_b3(m, base, static_cast<uint64_t>(ncols), static_cast<uint64_t>(K))
               : make_map(m, base, static_cast<uint64_t>(ncols), static_cast<uint64_t>(K), 64, 64);
}

// fp32 [outer x inner] row-major, box {32, 32} with 128-byte swizzle: the
// target of the reduce-add form's tile reductions.
int make_map_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer)
{
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool act_ok(int a) { return a == TFFN_ACT_NONE || a == TFFN_ACT_RELU || a == TFFN_ACT_GELU_TANH || a == TFFN_ACT_SILU; }
bool dim_ok(int64_t d) { return d >= 8 && d % 8 == 0 && d < (int64_t(1) << 31); }

// Current device's state, initialised on first use.
int device_state(DeviceState** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return TFFN_ERR_CUDA;
    DeviceState& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TFFN_ERR_CUDA;
        if (get_encode() != 0)
            return TFFN_ERR_CUDA;
        d.init = true;
    }
    *out = &d;
    return TFFN_OK;
}

// Workspace of at least `need` bytes, initialised; returns its base.
int workspace(DeviceState& d, size_t need, cudaStream_t s, uint8_t** base)
{
    void* b = nullptr;
    if (d.user_set) {
        if (d.user_bytes < need)
            return TFFN_ERR_NO_WORKSPACE;
        b = d.user;
    } else {
        if (d.owned_bytes < need) {
            if (d.owned) {
                if (cudaFree(d.owned) != cudaSuccess)
                    return TFFN_ERR_CUDA;
                d.owned = nullptr;
                d.owned_bytes = 0;
            }
            const size_t bytes = align_up(need, size_t(64) << 20);
            if (cudaMalloc(&d.owned, bytes) != cudaSuccess) {
                d.owned = nullptr;
                return TFFN_ERR_CUDA;
            }
            d.owned_bytes = bytes;
            d.needs_reset = true;
        }
        b = d.owned;
    }
    if (d.needs_reset) {
        if (cudaMemsetAsync(b, 0, SYNC_BYTES, s) != cudaSuccess)
            return TFFN_ERR_CUDA;
        d.launches = 0;
        d.needs_reset = false;
    }
    *base = static_cast<uint8_t*>(b);
    return TFFN_OK;
}

// Ready flags hold the epoch of the launch that stamped them, and the epoch
// lives in the control block (each launch uses the stored value + 1).  The
// host only counts launches so that, long before the 32-bit epoch could wrap,
// the flag region is cleared again.
int count_launch(DeviceState& d, uint8_t* base, cudaStream_t s)
{
    if (++d.launches >= EPOCH_LIMIT) {
        if (cudaMemsetAsync(base, 0, SYNC_BYTES, s) != cudaSuccess)
            return TFFN_ERR_CUDA;
        d.launches = 1;
    }
    return TFFN_OK;
}

void timing_start(cudaStream_t s)
{
    g_timing_this = g_timing && (g_timing_seen++ % static_cast<uint64_t>(g_timing_every)) == 0;
    if (!g_timing_this)
        return;
    if (g_events_used == g_events.size()) {
        cudaEvent_t a, b;
        cudaEventCreate(&a);
        cudaEventCreate(&b);
        g_events.emplace_back(a, b);
    }
    cudaEventRecord(g_events[g_events_used].first, s);
}

void timing_stop(cudaStream_t s)
{
    if (!g_timing_this)
        return;
    g_timing_this = false;
    cudaEventRecord(g_events[g_events_used].second, s);
    ++g_events_used;
}

// Row bands per raster group of the engine.  Inside a group the tiles go
// column by column, so the CTA pairs in flight read (pairs / group) weight
// panels of N x 256 at a time; on GB300 both measured optima hold ~38 MB of
// panels in flight: 4 bands at N 4096 (prefill: 0.731 ms against 0.749-0.762
// at 2, 8 or 16), 8 bands at N 8192 (large: 9.61 ms against 9.71-9.77 at 4
// and 9.81-9.87 at 16).  TFFN_OPT_GROUP_M > 0 overrides.
int32_t raster_group(int64_t N)
{
    const int64_t g = g_opt_group.load();
    if (g > 0)
        return static_cast<int32_t>(g);
    return N >= 8192 ? 8 : 4;
}

uint64_t wait_limit_ns()
{
    int64_t ms = g_opt_wait_ms.load();
    if (ms < 1)
        ms = 1;
    return static_cast<uint64_t>(ms) * 1000000ull;
}

// ------------------------------------------------------------------ layouts
struct DenseLayout {
    int path = 0;          // 1 engine fused, 2 decode, 3 engine two launches, 4 reduce-add form,
                           // 5 back-to-back (H on chip), 6 tensor-core weight stream
    int64_t m_blocks = 0;
    int32_t n1 = 0, n2 = 0;
    size_t off_h = 0;      // engine: H [m_blocks*BM x O]; decode: H [M x O]
    size_t off_part = 0;   // decode and tensor-core stream: split-K partial sums
    size_t total = 0;
};

// glu: the gated form, whose layer-1 engine tiles cover 128 hidden columns
// each (and decode slices 64).  sms: the CTA count the decode launch plans
// for (its split-K partial area depends on it).
DenseLayout dense_layout(int64_t M, int64_t N, int64_t O, int64_t P, int sms, bool glu = false)
{
    DenseLayout L;
    int64_t path = g_opt_path.load();
    if (path == 0) {
        if (M <= DECODE_MAX_M)
            path = 2;
        else if (M <= STREAM_MAX_M)
            path = 6;
        else if (M <= wstream::MAX_ROWS && wstream::make_plan(M, N, O, P, sms, glu).win == 1)
            path = 6;   // on the Llama 3 8B shape at 256 rows: 87 us against 125 us on the engine (with
                        // four-block windows, (8192, 28672, 8192) at 256 rows: 247 us against 236)
        else
            path = 1;
    }
    if (path == 2 && M > decode::MAX_ROWS)
        path = 1;
    if (path == 6 && M > wstream::MAX_ROWS)
        path = 1;
    if ((path == 4 || path == 5) && glu)
        path = 1;
    L.path = static_cast<int>(path);
    L.off_h = SYNC_BYTES;
    if (L.path == 4) {
        // the reduce-add form: an fp32 accumulator of Y instead of H; one
        // counter per 32-row strip of each Y tile in the flag region
        L.m_blocks = (M + engine::BM - 1) / engine::BM;
        L.n1 = static_cast<int32_t>((O + engine::BN - 1) / engine::BN);
        L.n2 = static_cast<int32_t>((P + engine::BN - 1) / engine::BN);
        if (static_cast<size_t>(L.m_blocks) * L.n2 * reduce::COUNTERS_PER_TILE <= FLAG_WORDS) {
            L.total = align_up(L.off_h + static_cast<size_t>(L.m_blocks) * engine::BM * P * 4, 256);
            return L;
        }
        L.path = 1;
    }
    if (L.path == 5) {
        // back-to-back: nothing but the control block
        L.m_blocks = (M + engine::BM - 1) / engine::BM;
        L.n1 = static_cast<int32_t>((O + engine::BN - 1) / engine::BN);
        L.n2 = static_cast<int32_t>((P + engine::BN - 1) / engine::BN);
        L.total = SYNC_BYTES;
        return L;
    }
    if (L.path == 2) {
        const decode::Plan pl = decode::make_plan(M, N, O, P, sms, glu);
        L.off_part = align_up(L.off_h + static_cast<size_t>(M) * O * 2, 256);
        L.total = L.off_part + pl.partial_bytes;
        return L;
    }
    if (L.path == 6) {
        const wstream::Plan pl = wstream::make_plan(M, N, O, P, sms, glu);
        L.off_part = align_up(L.off_h + static_cast<size_t>(M) * O * 2, 256);
        L.total = L.off_part + pl.partial_bytes;
        return L;
    }
    L.m_blocks = (M + engine::BM - 1) / engine::BM;
    const int64_t h_cols = glu ? engine::BN_CTA : engine::BN;   // hidden columns per layer-1 tile
    L.n1 = static_cast<int32_t>((O + h_cols - 1) / h_cols);
    L.n2 = static_cast<int32_t>((P + engine::BN - 1) / engine::BN);
    if (L.path == 1 && static_cast<size_t>(L.m_blocks) * L.n1 * engine::FLAG_WORDS_PER_TILE > FLAG_WORDS)
        L.path = 3;   // more layer-1 tiles than flags: run the layers as two launches
    L.total = align_up(L.off_h + static_cast<size_t>(L.m_blocks) * engine::BM * O * 2, 256);
    return L;
}

struct MoeLayout {
    int64_t R = 0, Rmax = 0, mbmax = 0;
    int32_t n1 = 0, n2 = 0;
    size_t off_idx, off_w, off_pos, off_hist, off_bpad, off_boff, off_pad, off_band, off_nb, off_rowent, off_xp,
        off_h, off_yp, total;
};

// glu: gated experts, whose layer-1 tiles cover 128 hidden columns
MoeLayout moe_layout(int64_t T, int64_t N, int64_t O, int64_t P, int E, int k, bool glu = false)
{
    MoeLayout L;
    L.R = T * k;
    L.Rmax = static_cast<int64_t>(align_up(static_cast<size_t>(L.R + static_cast<int64_t>(E) * (engine::BM - 1)),
                                           engine::BM));
    L.mbmax = L.Rmax / engine::BM;
    const int64_t h_cols = glu ? engine::BN_CTA : engine::BN;
    L.n1 = static_cast<int32_t>((O + h_cols - 1) / h_cols);
    L.n2 = static_cast<int32_t>((P + engine::BN - 1) / engine::BN);
    size_t o = SYNC_BYTES;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.off_idx = take(static_cast<size_t>(L.R) * 4);
    L.off_w = take(static_cast<size_t>(L.R) * 4);
    L.off_pos = take(static_cast<size_t>(L.R) * 4);
    const size_t blk_words = static_cast<size_t>(moe_route_blocks(T)) * E;   // per token block, per expert
    L.off_hist = take(blk_words * 4);
    L.off_bpad = take(blk_words * 4);
    L.off_boff = take(blk_words * 4);
    L.off_pad = take(static_cast<size_t>(2 * E) * 4);
    L.off_band = take(static_cast<size_t>(L.mbmax) * 4);
    L.off_nb = take(4);
    L.off_rowent = take(static_cast<size_t>(L.Rmax) * 4);
    L.off_xp = take(static_cast<size_t>(L.Rmax) * N * 2);
    L.off_h = take(static_cast<size_t>(L.Rmax) * O * 2);
    L.off_yp = take(static_cast<size_t>(L.Rmax) * P * 4);
    L.total = o;
    return L;
}

template <int MAX_E>
void fill_layer(engine::LayerArgs& la, int64_t K, int64_t ncols, int act, int out_f32, int64_t rows, void* out)
{
    la.K = static_cast<int32_t>(K);
    la.ncols = static_cast<int32_t>(ncols);
    la.n_tiles = static_cast<int32_t>((ncols + engine::BN - 1) / engine::BN);
    la.act = act;
    la.out_f32 = out_f32;
    la.pad_ = 0;
    la.ld_out = ncols;
    la.rows = rows;
    la.out = out;
}

}  // namespace

namespace tffn {
uint64_t option_wait_limit_ns() { return wait_limit_ns(); }
int32_t option_skip_flag() { return static_cast<int32_t>(g_opt_skip.load()); }
}  // namespace tffn

// Key of a dense-FFN call: everything its kernel parameters depend on.
static CallKey dense_key(int kind, int path, const void* X, const void* W1, const void* W3, const void* b1,
                         const void* W2, const void* b2, void* Y, const uint8_t* base, int act1, int act2,
                         int64_t M, int64_t N, int64_t O, int64_t P, int sms)
{
    CallKey k;
    k.kind = kind;
    k.path = path;
    k.act1 = act1;
    k.act2 = act2;
    k.dims[0] = M;
    k.dims[1] = N;
    k.dims[2] = O;
    k.dims[3] = P;
    k.dims[4] = sms;
    k.ptrs = {X, W1, W3, b1, W2, b2, Y, base};
    return k;
}

// The weight-streaming decode launch (dense, or gated when W3 is given).
static int run_decode(DeviceState& d, uint8_t* base, const DenseLayout& L, const void* X, const void* W1,
                      const void* W3, const void* b1, const void* W2, const void* b2, int act1, int act2, int64_t M,
                      int64_t N, int64_t O, int64_t P, void* Y, cudaStream_t s)
{
    int rc = count_launch(d, base, s);
    if (rc != TFFN_OK)
        return rc;
    const bool glu = W3 != nullptr;
    const CallKey key = dense_key(2, L.path, X, W1, W3, b1, W2, b2, Y, base, act1, act2, M, N, O, P, d.sms);
    decode::Params* cp = d.decode_cache.find(key);
    if (cp == nullptr) {
        decode::Params p{};
        p.X = static_cast<const __nv_bfloat16*>(X);
        p.W1 = static_cast<const __nv_bfloat16*>(W1);
        p.b1 = static_cast<const __nv_bfloat16*>(b1);
        p.W2 = static_cast<const __nv_bfloat16*>(W2);
        p.b2 = static_cast<const __nv_bfloat16*>(b2);
        p.Y = static_cast<__nv_bfloat16*>(Y);
        p.H = reinterpret_cast<__nv_bfloat16*>(base + L.off_h);
        p.partial = reinterpret_cast<float*>(base + L.off_part);
        p.counters = reinterpret_cast<uint32_t*>(base + OFF_DCOUNT);
        p.flags = reinterpret_cast<uint32_t*>(base + OFF_FLAGS);
        p.ctrl = reinterpret_cast<DevCtrl*>(base);
        p.M = static_cast<int32_t>(M);
        p.N = static_cast<int32_t>(N);
        p.O = static_cast<int32_t>(O);
        p.P = static_cast<int32_t>(P);
        p.act1 = act1;
        p.act2 = act2;
        p.glu = glu ? 1 : 0;
        p.plan = decode::make_plan(M, N, O, P, d.sms, glu);
        if (static_cast<size_t>(p.plan.slices[0]) * 4 > FLAG_WORDS ||
            (static_cast<size_t>(p.plan.slices[0]) + p.plan.slices[1]) * 4 > DCOUNT_WORDS)
            return TFFN_ERR_UNSUPPORTED;
        const uint32_t arows = M <= 16 ? 16u : static_cast<uint32_t>(decode::decode_rows(M));
        // Gated layer 1 loads 64-column boxes of W1 and W3 (128 B per row) whose
        // neighbours belong to other units: no promotion past 128 B, or every
        // weight row would be fetched twice.
        const CUtensorMapL2promotion w1_promo =
            glu ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
        // the gated window reads 128 adjacent columns of W1 and of W3 per row
        // (two boxes each): 256-byte promotion, boxes of KC1 rows
        const uint32_t w1_rows =
            p.plan.win ? static_cast<uint32_t>(decode::KC1) : static_cast<uint32_t>(decode::KC);
        const CUtensorMapL2promotion w1p = p.plan.win ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : w1_promo;
        if (make_map(&p.map_w[0], W1, O, N, 64, w1_rows, w1p) ||
            make_map(&p.map_w[1], W2, P, O, 64, decode::KC) || make_map(&p.map_a[0], X, N, M, 64, arows) ||
            make_map(&p.map_a[1], p.H, O, M, 64, arows) ||
            (glu && make_map(&p.map_w3, W3, O, N, 64, w1_rows, w1p)))
            return TFFN_ERR_INVALID_ARG;
        cp = d.decode_cache.store(key, p);
    }
    cp->skip_slice = glu ? -1 : static_cast<int32_t>(g_opt_skip.load());
    cp->wait_limit_ns = wait_limit_ns();
    timing_start(s);
    if (launch_decode(*cp, cp->plan.grid, s) != 0)
        return TFFN_ERR_CUDA;
    timing_stop(s);
    g_last_launches = 1;
    return TFFN_OK;
}

// The tensor-core weight stream (dense, or gated when W3 is given).
static int run_wstream(DeviceState& d, uint8_t* base, const DenseLayout& L, const void* X, const void* W1,
                       const void* W3, const void* b1, const void* W2, const void* b2, int act1, int act2,
                       int64_t M, int64_t N, int64_t O, int64_t P, void* Y, cudaStream_t s)
{
    int rc = count_launch(d, base, s);
    if (rc != TFFN_OK)
        return rc;
    const bool glu = W3 != nullptr;
    const CallKey key = dense_key(6, L.path, X, W1, W3, b1, W2, b2, Y, base, act1, act2, M, N, O, P, d.sms);
    wstream::Params* cp = d.wstream_cache.find(key);
    if (cp == nullptr) {
        wstream::Params p{};
        p.b1 = static_cast<const __nv_bfloat16*>(b1);
        p.b2 = static_cast<const __nv_bfloat16*>(b2);
        p.Y = static_cast<__nv_bfloat16*>(Y);
        p.H = reinterpret_cast<__nv_bfloat16*>(base + L.off_h);
        p.partial = reinterpret_cast<float*>(base + L.off_part);
        p.counters = reinterpret_cast<uint32_t*>(base + OFF_DCOUNT);
        p.flags = reinterpret_cast<uint32_t*>(base + OFF_FLAGS);
        p.ctrl = reinterpret_cast<DevCtrl*>(base);
        p.M = static_cast<int32_t>(M);
        p.N = static_cast<int32_t>(N);
        p.O = static_cast<int32_t>(O);
        p.P = static_cast<int32_t>(P);
        p.act1 = act1;
        p.act2 = act2;
        p.glu = glu ? 1 : 0;
        p.plan = wstream::make_plan(M, N, O, P, d.sms, glu);
        const size_t flag_words = p.plan.win ? static_cast<size_t>(p.plan.nblk) * 2
                                             : static_cast<size_t>(p.plan.slices[0]) * wstream::EPI_WARPS;
        if (flag_words > FLAG_WORDS ||
            2 * (static_cast<size_t>(p.plan.slices[0]) + p.plan.slices[1]) * wstream::EPI_WARPS > DCOUNT_WORDS)
            return TFFN_ERR_UNSUPPORTED;
        const uint32_t rows = static_cast<uint32_t>(p.plan.rows);
        if (make_map(&p.map_w[0], W1, O, N, 64, wstream::KC) || make_map(&p.map_w[1], W2, P, O, 64, wstream::KC) ||
            make_map(&p.map_x[0], X, N, M, 64, rows) || make_map(&p.map_x[1], p.H, O, M, 64, rows) ||
            (glu && make_map(&p.map_w3, W3, O, N, 64, wstream::KC)))
            return TFFN_ERR_INVALID_ARG;
        cp = d.wstream_cache.store(key, p);
    }
    cp->wait_limit_ns = wait_limit_ns();
    timing_start(s);
    if (launch_wstream(*cp, s) != 0)
        return TFFN_ERR_CUDA;
    timing_stop(s);
    g_last_launches = 1;
    return TFFN_OK;
}

// Launch the dense engine as the layout says: one fused launch, or layer 1
// and layer 2 as two launches.
static int run_dense_engine(DeviceState& d, uint8_t* base, const DenseLayout& L, engine::Params<1>& p,
                            cudaStream_t s)
{
    if (engine_total_tickets(L.m_blocks, L.n1, L.n2, MODE_FUSED) > ENGINE_MAX_TICKETS)
        return TFFN_ERR_INVALID_ARG;
    p.layer[0].n_tiles = L.n1;
    p.m_blocks = L.m_blocks;
    p.m_blocks_dev = nullptr;
    p.band_expert = nullptr;
    p.flags = reinterpret_cast<uint32_t*>(base + OFF_FLAGS);
    p.band_count = band_counts(base, L.m_blocks);
    p.ctrl = reinterpret_cast<DevCtrl*>(base);
    p.wait_limit_ns = wait_limit_ns();
    p.group_m = raster_group(p.layer[0].K);
    p.skip_flag = static_cast<int32_t>(g_opt_skip.load());
    if (L.path == 1) {
        int rc = count_launch(d, base, s);
        if (rc != TFFN_OK)
            return rc;
        p.mode = MODE_FUSED;
        const int64_t total = engine_total_tickets(L.m_blocks, L.n1, L.n2, MODE_FUSED);
        const int pairs = static_cast<int>(total < d.sms ? total : d.sms);
        timing_start(s);
        if (launch_engine_dense(p, pairs, s) != 0)
            return TFFN_ERR_CUDA;
        timing_stop(s);
        g_last_launches = 1;
        return TFFN_OK;
    }
    for (int mode = MODE_LAYER1; mode <= MODE_LAYER2; ++mode) {
        p.mode = mode;
        const int64_t total = engine_total_tickets(L.m_blocks, L.n1, L.n2, mode);
        const int pairs = static_cast<int>(total < d.sms ? total : d.sms);
        if (mode == MODE_LAYER1)
            timing_start(s);
        if (launch_engine_dense(p, pairs, s) != 0)
            return TFFN_ERR_CUDA;
        ++g_last_launches;
    }
    timing_stop(s);
    return TFFN_OK;
}

// ====================================================================== ABI

extern "C" {

int ffn_forward(const void* X, const void* W1, const void* b1, const void* W2, const void* b2, int act1,
                int act2, int64_t M, int64_t N, int64_t O, int64_t P, void* Y, struct CUstream_st* stream)
{
    g_last_launches = 0;
    if (M < 0 || M >= (int64_t(1) << 31) || !dim_ok(N) || !dim_ok(O) || !dim_ok(P))
        return TFFN_ERR_INVALID_ARG;
    if (!act_ok(act1) || !act_ok(act2))
        return TFFN_ERR_INVALID_ARG;
    if (M == 0)
        return TFFN_OK;   // empty call: X and Y may be NULL
    if (!X || !W1 || !W2 || !Y)
        return TFFN_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W2) || !aligned16(Y) || (b1 && !aligned16(b1)) ||
        (b2 && !aligned16(b2)))
        return TFFN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != TFFN_OK)
        return rc;
    const DenseLayout L = dense_layout(M, N, O, P, d->sms);
    uint8_t* base = nullptr;
    rc = workspace(*d, L.total, s, &base);
    if (rc != TFFN_OK)
        return rc;
    DevCtrl* ctrl = reinterpret_cast<DevCtrl*>(base);
    uint32_t* flags = reinterpret_cast<uint32_t*>(base + OFF_FLAGS);

    if (L.path == 2)
        return run_decode(*d, base, L, X, W1, nullptr, b1, W2, b2, act1, act2, M, N, O, P, Y, s);
    if (L.path == 6)
        return run_wstream(*d, base, L, X, W1, nullptr, b1, W2, b2, act1, act2, M, N, O, P, Y, s);

    if (L.path == 4 || L.path == 5) {
        reduce::Params rp;
        std::memset(&rp, 0, sizeof(rp));
        float* acc = reinterpret_cast<float*>(base + L.off_h);
        const int64_t rows_acc = L.m_blocks * engine::BM;
        const bool b3d = (O % 64 == 0) && (P % 64 == 0);
        if (make_map(&rp.map_x, X, N, M, 64, engine::BM_CTA) || make_map_b(&rp.map_w1, W1, O, N, b3d) ||
            make_map_b(&rp.map_w2, W2, P, O, b3d) || (L.path == 4 && make_map_f32(&rp.map_acc, acc, P, rows_acc)))
            return TFFN_ERR_INVALID_ARG;
        rp.b1 = static_cast<const __nv_bfloat16*>(b1);
        rp.b2 = static_cast<const __nv_bfloat16*>(b2);
        rp.acc = acc;
        rp.Y = static_cast<__nv_bfloat16*>(Y);
        rp.counters = flags;
        rp.ctrl = ctrl;
        rp.wait_limit_ns = wait_limit_ns();
        rp.M = M;
        rp.N = static_cast<int32_t>(N);
        rp.O = static_cast<int32_t>(O);
        rp.P = static_cast<int32_t>(P);
        rp.act1 = act1;
        rp.act2 = act2;
        rp.m_blocks = static_cast<int32_t>(L.m_blocks);
        rp.n_h = L.n1;
        rp.n_p = L.n2;
        rp.b3d = b3d ? 1 : 0;
        if (L.path == 5) {   // one task per (band, Y tile)
            const int64_t total = L.m_blocks * static_cast<int64_t>(L.n2);
            const int pairs = static_cast<int>(total < d->sms ? total : d->sms);
            timing_start(s);
            if (launch_b2b(rp, pairs, s) != 0)
                return TFFN_ERR_CUDA;
            timing_stop(s);
            g_last_launches = 1;
            return TFFN_OK;
        }
        // the counters and the accumulator start at zero in every call
        const size_t counter_bytes = static_cast<size_t>(L.m_blocks) * L.n2 * reduce::COUNTERS_PER_TILE * 4;
        if (cudaMemsetAsync(flags, 0, counter_bytes, s) != cudaSuccess ||
            cudaMemsetAsync(acc, 0, static_cast<size_t>(rows_acc) * P * 4, s) != cudaSuccess)
            return TFFN_ERR_CUDA;
        const int64_t total = L.m_blocks * static_cast<int64_t>(L.n1);
        const int pairs = static_cast<int>(total < d->sms ? total : d->sms);
        timing_start(s);
        if (launch_reduce(rp, pairs, s) != 0)
            return TFFN_ERR_CUDA;
        timing_stop(s);
        g_last_launches = 1;
        return TFFN_OK;
    }

    const CallKey key = dense_key(1, L.path, X, W1, nullptr, b1, W2, b2, Y, base, act1, act2, M, N, O, P, d->sms);
    engine::Params<1>* cp = d->engine_cache.find(key);
    if (cp == nullptr) {
        engine::Params<1> p;
        std::memset(&p, 0, sizeof(p));
        void* H = base + L.off_h;
        const int64_t rows_h = L.m_blocks * engine::BM;
        const bool b3d = (O % 64 == 0) && (P % 64 == 0);
        if (make_map(&p.map_a[0], X, N, M, 64, engine::BM_CTA) ||
            make_map(&p.map_a[1], H, O, rows_h, 64, engine::BM_CTA) || make_map_b(&p.map_b[0][0], W1, O, N, b3d) ||
            make_map_b(&p.map_b[1][0], W2, P, O, b3d) ||
            make_map(&p.map_out[0], H, O, rows_h, engine::OUT_COLS, 32) ||
            make_map(&p.map_out[1], Y, P, M, engine::OUT_COLS, 32))
            return TFFN_ERR_INVALID_ARG;
        p.b3d = b3d ? 1 : 0;
        p.bias[0][0] = static_cast<const __nv_bfloat16*>(b1);
        p.bias[1][0] = static_cast<const __nv_bfloat16*>(b2);
        fill_layer<1>(p.layer[0], N, O, act1, 0, rows_h, H);
        fill_layer<1>(p.layer[1], O, P, act2, 0, M, Y);
        cp = d->engine_cache.store(key, p);
    }
    return run_dense_engine(*d, base, L, *cp, s);
}

int ffn_glu_forward(const void* X, const void* W1, const void* W3, const void* W2, int act, int64_t M, int64_t N,
                    int64_t O, int64_t P, void* Y, struct CUstream_st* stream)
{
    g_last_launches = 0;
    if (M < 0 || M >= (int64_t(1) << 31) || !dim_ok(N) || !dim_ok(O) || !dim_ok(P) || !act_ok(act))
        return TFFN_ERR_INVALID_ARG;
    if (M == 0)
        return TFFN_OK;   // empty call: X and Y may be NULL
    if (!X || !W1 || !W3 || !W2 || !Y)
        return TFFN_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(Y))
        return TFFN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != TFFN_OK)
        return rc;
    const DenseLayout L = dense_layout(M, N, O, P, d->sms, true);
    uint8_t* base = nullptr;
    rc = workspace(*d, L.total, s, &base);
    if (rc != TFFN_OK)
        return rc;
    if (L.path == 2)
        return run_decode(*d, base, L, X, W1, W3, nullptr, W2, nullptr, act, TFFN_ACT_NONE, M, N, O, P, Y, s);
    if (L.path == 6)
        return run_wstream(*d, base, L, X, W1, W3, nullptr, W2, nullptr, act, TFFN_ACT_NONE, M, N, O, P, Y, s);

    const CallKey key =
        dense_key(11, L.path, X, W1, W3, nullptr, W2, nullptr, Y, base, act, TFFN_ACT_NONE, M, N, O, P, d->sms);
    engine::Params<1>* cp = d->engine_cache.find(key);
    if (cp == nullptr) {
        engine::Params<1> p;
        std::memset(&p, 0, sizeof(p));
        void* H = base + L.off_h;
        const int64_t rows_h = L.m_blocks * engine::BM;
        const bool b3d = (O % 64 == 0) && (P % 64 == 0);
        if (make_map(&p.map_a[0], X, N, M, 64, engine::BM_CTA) ||
            make_map(&p.map_a[1], H, O, rows_h, 64, engine::BM_CTA) || make_map_b(&p.map_b[0][0], W1, O, N, b3d) ||
            make_map_b(&p.map_b_lin[0], W3, O, N, b3d) || make_map_b(&p.map_b[1][0], W2, P, O, b3d) ||
            make_map(&p.map_out[0], H, O, rows_h, engine::OUT_COLS, 32) ||
            make_map(&p.map_out[1], Y, P, M, engine::OUT_COLS, 32))
            return TFFN_ERR_INVALID_ARG;
        p.b3d = b3d ? 1 : 0;
        p.glu = 1;
        fill_layer<1>(p.layer[0], N, O, act, 0, rows_h, H);
        fill_layer<1>(p.layer[1], O, P, TFFN_ACT_NONE, 0, M, Y);
        cp = d->engine_cache.store(key, p);
    }
    return run_dense_engine(*d, base, L, *cp, s);
}

// The MoE forward; W3 (an array of E pointers) non-null: gated experts.
static int moe_forward(const void* X, const float* gate_logits, int top_k, const void* const* W1,
                       const void* const* W3, const void* const* b1, const void* const* W2, const void* const* b2,
                       void* Y, int64_t T, int64_t N, int64_t O, int64_t P, int E, int act1, int act2,
                       tffn_routing* routing, struct CUstream_st* stream)
{
    g_last_launches = 0;
    const bool glu = W3 != nullptr;
    if (E < 1 || E > MOE_MAX_E || top_k < 1 || top_k > E)
        return TFFN_ERR_INVALID_ARG;
    if (T < 0 || T * top_k >= (int64_t(1) << 30) || !dim_ok(N) || !dim_ok(O) || !dim_ok(P))
        return TFFN_ERR_INVALID_ARG;
    if (!act_ok(act1) || !act_ok(act2))
        return TFFN_ERR_INVALID_ARG;
    if (T == 0)
        return TFFN_OK;   // empty call: X, gate_logits and Y may be NULL
    if (!X || !gate_logits || !W1 || !W2 || !Y)
        return TFFN_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(gate_logits) & 3u))
        return TFFN_ERR_INVALID_ARG;
    for (int e = 0; e < E; ++e) {
        if (!W1[e] || !W2[e] || !aligned16(W1[e]) || !aligned16(W2[e]))
            return TFFN_ERR_INVALID_ARG;
        if (glu && (!W3[e] || !aligned16(W3[e])))
            return TFFN_ERR_INVALID_ARG;
        if (b1 && b1[e] && !aligned16(b1[e]))
            return TFFN_ERR_INVALID_ARG;
        if (b2 && b2[e] && !aligned16(b2[e]))
            return TFFN_ERR_INVALID_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != TFFN_OK)
        return rc;
    const MoeLayout L = moe_layout(T, N, O, P, E, top_k, glu);
    if (static_cast<size_t>(L.mbmax) * L.n1 * engine::FLAG_WORDS_PER_TILE > FLAG_WORDS)
        return TFFN_ERR_UNSUPPORTED;
    uint8_t* base = nullptr;
    rc = workspace(*d, L.total, s, &base);
    if (rc != TFFN_OK)
        return rc;
    if ((rc = count_launch(*d, base, s)) != TFFN_OK)
        return rc;

    int32_t* idx = reinterpret_cast<int32_t*>(base + L.off_idx);
    float* w = reinterpret_cast<float*>(base + L.off_w);
    int32_t* pos = reinterpret_cast<int32_t*>(base + L.off_pos);
    int32_t* hist = reinterpret_cast<int32_t*>(base + L.off_hist);
    int32_t* bpad = reinterpret_cast<int32_t*>(base + L.off_bpad);
    int32_t* boff = reinterpret_cast<int32_t*>(base + L.off_boff);
    int32_t* padt = reinterpret_cast<int32_t*>(base + L.off_pad);
    int32_t* band = reinterpret_cast<int32_t*>(base + L.off_band);
    int32_t* nb = reinterpret_cast<int32_t*>(base + L.off_nb);
    int32_t* rowent = reinterpret_cast<int32_t*>(base + L.off_rowent);
    void* Xp = base + L.off_xp;
    void* H = base + L.off_h;
    float* Yp = reinterpret_cast<float*>(base + L.off_yp);
    // The weighted sum of the experts' outputs runs in the engine's layer-2
    // epilogue when the per-token counters fit the sync region (else, or with
    // TFFN_OPT_MOE_COMBINE = 0, as a separate kernel; identical results).
    const bool fused_combine = g_opt_moe_combine.load() != 0 &&
                               static_cast<size_t>(T) * static_cast<size_t>(L.n2) <= MCOUNT_WORDS;

    CallKey key;
    key.kind = glu ? 65 : 64;
    key.act1 = act1;
    key.act2 = act2;
    key.dims[0] = T;
    key.dims[1] = N;
    key.dims[2] = O;
    key.dims[3] = P;
    key.dims[4] = E;
    key.dims[5] = top_k;
    key.ptrs.reserve(2 + 5 * static_cast<size_t>(E));
    key.ptrs.push_back(base);
    key.ptrs.push_back(Y);
    for (int e = 0; e < E; ++e) {
        key.ptrs.push_back(W1[e]);
        key.ptrs.push_back(W2[e]);
        key.ptrs.push_back(glu ? W3[e] : nullptr);
        key.ptrs.push_back(b1 ? b1[e] : nullptr);
        key.ptrs.push_back(b2 ? b2[e] : nullptr);
    }
    engine::Params<MOE_MAX_E>* cp = d->moe_cache.find(key);
    if (cp == nullptr) {
        std::unique_ptr<engine::Params<MOE_MAX_E>> pp(new engine::Params<MOE_MAX_E>);
        std::memset(static_cast<void*>(pp.get()), 0, sizeof(*pp));
        engine::Params<MOE_MAX_E>& p = *pp;
        // outputs: H_perm (bf16, boxes of 32 rows x 64 columns) and the fp32
        // Y_perm (boxes of 32 rows x 32 columns, 128 bytes per row either way)
        int bad = make_map(&p.map_a[0], Xp, N, L.Rmax, 64, engine::BM_CTA) |
                  make_map(&p.map_a[1], H, O, L.Rmax, 64, engine::BM_CTA) |
                  make_map(&p.map_out[0], H, O, L.Rmax, engine::OUT_COLS, 32) |
                  make_map_f32(&p.map_out[1], Yp, P, L.Rmax);
        const bool b3d = (O % 64 == 0) && (P % 64 == 0);
        p.b3d = b3d ? 1 : 0;
        for (int e = 0; e < E && !bad; ++e) {
            bad |= make_map_b(&p.map_b[0][e], W1[e], O, N, b3d);
            bad |= make_map_b(&p.map_b[1][e], W2[e], P, O, b3d);
            if (glu)
                bad |= make_map_b(&p.map_b_lin[e], W3[e], O, N, b3d);
            p.bias[0][e] = b1 ? static_cast<const __nv_bfloat16*>(b1[e]) : nullptr;
            p.bias[1][e] = b2 ? static_cast<const __nv_bfloat16*>(b2[e]) : nullptr;
        }
        if (bad)
            return TFFN_ERR_INVALID_ARG;
        fill_layer<MOE_MAX_E>(p.layer[0], N, O, act1, 0, L.Rmax, H);
        fill_layer<MOE_MAX_E>(p.layer[1], O, P, act2, 1, L.Rmax, Yp);
        p.layer[0].n_tiles = L.n1;
        p.glu = glu ? 1 : 0;
        p.m_blocks = -1;
        p.m_blocks_dev = nb;
        p.band_expert = band;
        p.flags = reinterpret_cast<uint32_t*>(base + OFF_FLAGS);
        p.band_count = band_counts(base, L.mbmax);
        p.ctrl = reinterpret_cast<DevCtrl*>(base);
        p.mode = MODE_FUSED;
        cp = d->moe_cache.store(key, p);
    }
    engine::Params<MOE_MAX_E>& p = *cp;
    p.row_entry = fused_combine ? rowent : nullptr;
    p.comb_pos = pos;
    p.comb_w = w;
    p.comb_cnt = fused_combine ? reinterpret_cast<uint32_t*>(base + OFF_MCOUNT) : nullptr;
    p.comb_y = static_cast<__nv_bfloat16*>(Y);
    p.comb_k = top_k;
    p.wait_limit_ns = wait_limit_ns();
    p.group_m = raster_group(N);
    p.skip_flag = static_cast<int32_t>(g_opt_skip.load());

    if (engine_total_tickets(L.mbmax, L.n1, L.n2, MODE_FUSED) > ENGINE_MAX_TICKETS)
        return TFFN_ERR_INVALID_ARG;
    int fail = 0;
    fail |= launch_moe_route(gate_logits, T, E, top_k, idx, w, hist, s);
    fail |= launch_moe_plan(hist, T, E, engine::BM, g_opt_moe_order.load() != 0 ? 1 : 0, bpad, boff, band, nb, padt,
                            routing ? routing->expert_offsets : nullptr, s);
    fail |= launch_moe_scatter(idx, T, E, top_k, bpad, boff, pos, routing ? routing->perm : nullptr,
                               fused_combine ? rowent : nullptr, s);
    fail |= launch_moe_gather(X, pos, T, top_k, padt, E, N, Xp, fused_combine ? rowent : nullptr, d->sms * 4, s);
    if (!fail) {
        timing_start(s);
        fail |= launch_engine_grouped(p, d->sms / 2, s);
        timing_stop(s);
    }
    if (!fused_combine)
        fail |= launch_moe_combine(Yp, pos, w, T, top_k, P, Y, d->sms * 4, s);
    if (fail)
        return TFFN_ERR_CUDA;
    g_last_launches = fused_combine ? 5 : 6;
    if (routing && routing->topk_idx &&
        cudaMemcpyAsync(routing->topk_idx, idx, static_cast<size_t>(L.R) * 4, cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        return TFFN_ERR_CUDA;
    if (routing && routing->topk_w &&
        cudaMemcpyAsync(routing->topk_w, w, static_cast<size_t>(L.R) * 4, cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        return TFFN_ERR_CUDA;
    return TFFN_OK;
}

int moe_ffn_forward(const void* X, const float* gate_logits, int top_k, const void* const* W1,
                    const void* const* b1, const void* const* W2, const void* const* b2, void* Y, int64_t T,
                    int64_t N, int64_t O, int64_t P, int E, int act1, int act2, tffn_routing* routing,
                    struct CUstream_st* stream)
{
    return moe_forward(X, gate_logits, top_k, W1, nullptr, b1, W2, b2, Y, T, N, O, P, E, act1, act2, routing,
                       stream);
}

int moe_glu_forward(const void* X, const float* gate_logits, int top_k, const void* const* W1,
                    const void* const* W3, const void* const* W2, void* Y, int64_t T, int64_t N, int64_t O,
                    int64_t P, int E, int act, tffn_routing* routing, struct CUstream_st* stream)
{
    if (!W3 && T > 0)
        return TFFN_ERR_INVALID_ARG;
    return moe_forward(X, gate_logits, top_k, W1, W3, nullptr, W2, nullptr, Y, T, N, O, P, E, act, TFFN_ACT_NONE,
                       routing, stream);
}

size_t tffn_workspace_bytes(int64_t M, int64_t N, int64_t O, int64_t P, int E, int top_k)
{
    if (M < 0 || !dim_ok(N) || !dim_ok(O) || !dim_ok(P))
        return 0;
    if (E <= 0) {
        // the dense and the gated FFN, on the current device (or, without
        // one, planned for up to 1024 CTAs)
        int sms = 1024;
        DeviceState* d = nullptr;
        {
            std::lock_guard<std::mutex> lock(g_mu);
            if (device_state(&d) == TFFN_OK)
                sms = d->sms;
        }
        const size_t a = dense_layout(M, N, O, P, sms).total;
        const size_t b = dense_layout(M, N, O, P, sms, true).total;
        return a > b ? a : b;
    }
    if (top_k < 1 || top_k > E)
        return 0;
    return moe_layout(M, N, O, P, E, top_k).total;
}

int tffn_set_workspace(void* dev_ptr, size_t bytes)
{
    if (dev_ptr && ((reinterpret_cast<uintptr_t>(dev_ptr) & 255u) || bytes < SYNC_BYTES))
        return TFFN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return TFFN_ERR_CUDA;
    DeviceState& d = g_dev[dev];
    d.user = dev_ptr;
    d.user_bytes = dev_ptr ? bytes : 0;
    d.user_set = dev_ptr != nullptr;
    d.needs_reset = true;
    return TFFN_OK;
}

int tffn_check(struct CUstream_st* stream, int32_t* detail)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TFFN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return TFFN_ERR_CUDA;
    DeviceState& d = g_dev[dev];
    void* base = d.user_set ? d.user : d.owned;
    if (detail)
        detail[0] = detail[1] = detail[2] = detail[3] = 0;
    if (!base)
        return TFFN_OK;
    uint32_t rec[4] = {0, 0, 0, 0};
    if (cudaMemcpy(rec, base, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TFFN_ERR_CUDA;
    if (detail)
        for (int i = 0; i < 4; ++i)
            detail[i] = static_cast<int32_t>(rec[i]);
    if (rec[0] == 0)
        return TFFN_OK;
    // The failed launch may have left flags and counters inconsistent: the
    // whole sync region is re-zeroed before the next call.
    if (cudaMemset(base, 0, sizeof(rec)) != cudaSuccess)
        return TFFN_ERR_CUDA;
    d.needs_reset = true;
    const int32_t code = static_cast<int32_t>(rec[0]);
    return (code == TFFN_ERR_TIMEOUT) ? TFFN_ERR_TIMEOUT : TFFN_ERR_DEVICE;
}

const char* tffn_status_string(int status)
{
    switch (status) {
    case TFFN_OK: return "ok";
    case TFFN_ERR_INVALID_ARG: return "invalid argument";
    case TFFN_ERR_UNSUPPORTED: return "unsupported shape or option";
    case TFFN_ERR_CUDA: return "CUDA runtime error";
    case TFFN_ERR_TIMEOUT: return "device wait timed out";
    case TFFN_ERR_NO_WORKSPACE: return "workspace too small";
    case TFFN_ERR_DEVICE: return "device-side error";
    default: return "unknown status";
    }
}

int64_t tffn_set_option(int option, int64_t value)
{
    switch (option) {
    case TFFN_OPT_PATH: return (value < 0 || value > 6) ? -1 : g_opt_path.exchange(value);
    case TFFN_OPT_WAIT_LIMIT_MS: return g_opt_wait_ms.exchange(value);
    case TFFN_OPT_SKIP_FLAG: return g_opt_skip.exchange(value);
    case TFFN_OPT_GROUP_M: return g_opt_group.exchange(value);
    case TFFN_OPT_MOE_ORDER: return g_opt_moe_order.exchange(value);
    case TFFN_OPT_MOE_COMBINE: return g_opt_moe_combine.exchange(value);
    default: return -1;
    }
}

int tffn_last_launch_count(void) { return g_last_launches; }

int tffn_timing_begin(void)
{
    g_timing = true;
    g_events_used = 0;
    g_timing_seen = 0;
    return TFFN_OK;
}

int tffn_timing_sample(int every)
{
    if (every < 1)
        return TFFN_ERR_INVALID_ARG;
    g_timing_every = every;
    return TFFN_OK;
}

int tffn_timing_end(int* launches, double* total_ms)
{
    double sum = 0.0;
    for (size_t i = 0; i < g_events_used; ++i) {
        if (cudaEventSynchronize(g_events[i].second) != cudaSuccess)
            return TFFN_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, g_events[i].first, g_events[i].second) != cudaSuccess)
            return TFFN_ERR_CUDA;
        sum += ms;
    }
    if (launches)
        *launches = static_cast<int>(g_events_used);
    if (total_ms)
        *total_ms = sum;
    g_timing = false;
    g_events_used = 0;
    return TFFN_OK;
}

int64_t tffn_debug_engine_task(int64_t m_blocks, int32_t n1, int32_t n2, int32_t group_m, int64_t ticket,
                               int32_t out[3])
{
    if (group_m < 1)
        group_m = 1;
    const int64_t total = engine_total_tickets(m_blocks, n1, n2, MODE_FUSED);
    EngineTask t = engine_task(ticket, m_blocks, n1, n2, group_m, MODE_FUSED);
    if (ticket >= total)
        t.layer = -1;
    // The kernel maps tickets in 32-bit arithmetic: check it against this
    // 64-bit form wherever a launch may use it.
    if (total <= ENGINE_MAX_TICKETS && ticket >= 0 && ticket < ENGINE_MAX_TICKETS) {
        EngineTask t32 = engine_task_t<int32_t>(static_cast<int32_t>(ticket), static_cast<int32_t>(m_blocks), n1,
                                                n2, group_m, MODE_FUSED);
        if (ticket >= total)
            t32.layer = -1;
        if (t32.layer != t.layer || (t.layer >= 0 && (t32.band != t.band || t32.tile != t.tile)))
            return -1;
    }
    if (out) {
        out[0] = t.layer;
        out[1] = t.band;
        out[2] = t.tile;
    }
    return total;
}

void tffn_debug_tiles(int32_t out[6])
{
    out[0] = engine::BM;
    out[1] = engine::BN;
    out[2] = engine::BK;
    out[3] = engine::STAGES;
    out[4] = decode::SLICE;
    out[5] = decode::KC;
}

}  // extern "C"
