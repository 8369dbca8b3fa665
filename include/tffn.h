/*
 * tffn.h -- C ABI of the GB300-native fused Transformer FFN library.
 *
 * All tensors are dense row-major arrays in DEVICE memory of the current CUDA
 * device, owned by the caller; the library never frees them and keeps no
 * pointer to them after a call returns.  bf16 means IEEE bfloat16 (the upper
 * 16 bits of a binary32).  Calls are asynchronous on `stream` (a cudaStream_t;
 * NULL = legacy default stream): the return value covers argument validation
 * and launch errors only.  Errors found by a kernel while it runs (a wait that
 * timed out) are kept in the workspace and returned by tffn_check().
 *
 * Shapes and pointer rules shared by every entry point:
 *   - N, O, P are multiples of 8 and >= 8 (rows of every operand start on a
 *     16-byte boundary, as the tensor-memory-accelerator copies require);
 *   - every tensor pointer is 16-byte aligned;
 *   - M, T >= 0 (0 rows is a valid, empty call);
 *   - bias pointers may be NULL, meaning a zero bias.
 * A violation returns TFFN_ERR_INVALID_ARG before anything is launched.
 *
 * Workspace: the fused path keeps the hidden tensor H, ready flags and a
 * control block in a device workspace.  By default the library allocates it
 * (cudaMalloc, once per device, grown on demand; never inside a call that is
 * being captured into a CUDA graph if it has to grow).  A caller may instead
 * hand in its own buffer with tffn_set_workspace().  Calls that share a
 * workspace must be ordered on the GPU (same stream, or ordered by events).
 */
#ifndef TFFN_H
#define TFFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

/* Elementwise activations.  GELU is the tanh form
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))); SiLU (Swish with beta 1)
 * is x sigma(x) = x / (1 + exp(-x)). */
typedef enum {
    TFFN_ACT_NONE = 0,
    TFFN_ACT_RELU = 1,
    TFFN_ACT_GELU_TANH = 2,
    TFFN_ACT_SILU = 3
} tffn_act;

typedef enum {
    TFFN_OK = 0,
    TFFN_ERR_INVALID_ARG = -1,   /* bad pointer, size, alignment or code   */
    TFFN_ERR_UNSUPPORTED = -2,   /* valid, but outside what is implemented */
    TFFN_ERR_CUDA = -3,          /* a CUDA runtime call failed             */
    TFFN_ERR_TIMEOUT = -4,       /* a device-side wait ran out of time     */
    TFFN_ERR_NO_WORKSPACE = -5,  /* caller workspace too small             */
    TFFN_ERR_DEVICE = -6         /* other device-detected error            */
} tffn_status;

/*
 * ffn_forward -- Y = act2(act1(X W1 + b1) W2 + b2).
 *
 * Defined by "Kernel fusion and tensor parallelism" (brunomaga.github.io),
 * section "Megatron-LM tensor parallelism", the FFN equation: H is
 * act(X W1 + b1), Y is act(H W2 + b2), X in R^{MxN}, W1 in R^{NxO},
 * b1 in R^O, W2 in R^{OxP}, b2 in R^P; the second activation is optional
 * (TFFN_ACT_NONE), as Transformer FFNs omit it.  Section "Step 1" of the same
 * page fixes how the work is fused: each tile of H is multiplied by its row of
 * W2 tiles as soon as it is ready (Y_ik = sum_j H_ij (W2)_jk).
 *
 *   X  [M x N] bf16      W1 [N x O] bf16      b1 [O] bf16 (nullable)
 *   W2 [O x P] bf16      b2 [P] bf16 (nullable)
 *   Y  [M x P] bf16 (written; must not alias an input)
 *   act1, act2: tffn_act codes.
 *
 * Numerics: products accumulate in fp32; H is rounded to bf16 (round to
 * nearest even) after b1 and act1, as it is stored between the layers; Y is
 * rounded to bf16 after b2 and act2.
 * Paths: M <= 32 streams the weights with mma.sync (split-K, HBM-bound
 * decode shapes); 33 <= M <= 128 streams them with tcgen05 MMAs (the weights
 * as the MMA's M side, still HBM-bound), and so do 129 <= M <= 256 when every
 * CTA's share of the hidden width fits one 128-column window (O up to 128
 * times the SM count, two 64-column blocks per CTA); larger M runs the
 * persistent tcgen05 engine (GEMM1
 * tiles publish ready flags that GEMM2 tiles consume in the same launch).
 */
int ffn_forward(const void* X, const void* W1, const void* b1, const void* W2, const void* b2,
                int act1, int act2, int64_t M, int64_t N, int64_t O, int64_t P, void* Y,
                struct CUstream_st* stream);

/*
 * ffn_glu_forward -- gated FFN: Y = (act(X W1) * (X W3)) W2, * elementwise;
 * SwiGLU is act = TFFN_ACT_SILU (GeGLU: GELU, ReGLU: ReLU, bilinear: NONE).
 *
 * Defined by "Kernel fusion and tensor parallelism" (brunomaga.github.io),
 * section "Results": the SwiGLU FFN of the benchmarked models has a third
 * weight matrix, whose product with the input gates the activation, and no
 * biases.  The gate is the activated product X W1; X W3 multiplies it
 * (Shazeer, "GLU Variants Improve Transformer", 2020, equation for FFN_SwiGLU).
 *
 *   X  [M x N] bf16      W1 [N x O] bf16      W3 [N x O] bf16
 *   W2 [O x P] bf16      Y  [M x P] bf16 (written; must not alias an input)
 *   act: tffn_act code applied to X W1.
 *
 * Numerics: products accumulate in fp32; H = act(X W1) * (X W3) is rounded to
 * bf16 (nearest even) where it is stored between the layers; Y is rounded to
 * bf16.  Paths: M <= 32 streams the weights with mma.sync (each layer-1 unit
 * loads the same 64 columns of W1 and W3); 33 <= M <= 128 (up to 256 under
 * the same window condition as ffn_forward) streams them with tcgen05 MMAs
 * (gate and linear products in two tensor-memory accumulators); larger M
 * runs the persistent tcgen05 engine, each layer-1 tile pairing 128
 * columns of W1 with the same 128 columns of W3 in one 256-column
 * accumulator.  Errors and workspace as ffn_forward.
 */
int ffn_glu_forward(const void* X, const void* W1, const void* W3, const void* W2, int act, int64_t M,
                    int64_t N, int64_t O, int64_t P, void* Y, struct CUstream_st* stream);

/* Optional routing outputs of moe_ffn_forward (every member nullable; device
 * pointers): topk_idx[T*k] int32 and topk_w[T*k] fp32, slot s of token t at
 * t*k+s; perm[T*k] int32 maps the expert-grouped row r to t*k+s;
 * expert_offsets[E+1] int32 are the first grouped row of each expert. */
typedef struct {
    int32_t* topk_idx;
    float* topk_w;
    int32_t* perm;
    int32_t* expert_offsets;
} tffn_routing;

/*
 * moe_ffn_forward -- Mixture-of-Experts FFN: each token goes to its top_k
 * experts by gate logit; the output is the gate-weighted sum of those experts'
 * FFN outputs.
 *
 * Defined by "Fine-Grained Compute-Communication Overlap for MoE" (review of
 * arXiv 2607.19539, zhongzhuzhou.org), section 2.1 (the router's distribution
 * over E experts, top-k selection, gate-weighted sum) and section 2.2 steps 1,
 * 3 and 5 (routing, expert computation, weighted reduction); section 4.2 (rows
 * grouped contiguously per destination, each group zero-padded to a whole
 * tile) gives the grouped row layout; the expert FFN is ffn_forward's
 * ("Kernel fusion and tensor parallelism", section "Expert sharding").
 *
 *   X            [T x N] bf16
 *   gate_logits  [T x E] fp32
 *   W1, b1, W2, b2: HOST arrays of E DEVICE pointers; W1[e] [N x O],
 *                b1[e] [O] (array or entries nullable), W2[e] [O x P],
 *                b2[e] [P] (nullable) -- all bf16
 *   Y            [T x P] bf16 (written)
 *   1 <= top_k <= E <= 64.
 *
 * Routing: slot 0 holds the largest logit; equal logits go to the lower
 * expert index; the gate weights are the softmax over the top_k kept logits
 * (= softmax over E, keep top_k, renormalise to sum 1).  Each expert applies
 * its own b2 and act2 before the gate weighting; the weighted sum is taken in
 * fp32 in slot order and rounded to bf16 once.
 */
int moe_ffn_forward(const void* X, const float* gate_logits, int top_k, const void* const* W1,
                    const void* const* b1, const void* const* W2, const void* const* b2, void* Y,
                    int64_t T, int64_t N, int64_t O, int64_t P, int E, int act1, int act2,
                    tffn_routing* routing, struct CUstream_st* stream);

/*
 * moe_glu_forward -- moe_ffn_forward with gated experts: expert e computes
 * (act(x W1[e]) * (x W3[e])) W2[e] (ffn_glu_forward's FFN, no biases), as in
 * the SwiGLU experts of the MoE models the fused-FFN page benchmarks
 * ("Kernel fusion and tensor parallelism", sections "Expert sharding" and
 * "Results").  Routing, gate weights, grouping and the weighted sum are
 * moe_ffn_forward's.
 *
 *   W1, W3: HOST arrays of E DEVICE pointers, each [N x O] bf16
 *   W2:     HOST array of E DEVICE pointers, each [O x P] bf16
 *   act:    tffn_act code applied to x W1[e] (TFFN_ACT_SILU for SwiGLU)
 * Other arguments, errors and workspace as moe_ffn_forward (the workspace is
 * tffn_workspace_bytes(T, N, O, P, E, top_k)).
 */
int moe_glu_forward(const void* X, const float* gate_logits, int top_k, const void* const* W1,
                    const void* const* W3, const void* const* W2, void* Y, int64_t T, int64_t N, int64_t O,
                    int64_t P, int E, int act, tffn_routing* routing, struct CUstream_st* stream);

/*
 * ffn_forward_decode_noalloc -- ffn_forward for M <= 32 rows (the decode
 * shapes) that allocates nothing.  The paper has no counterpart: this entry
 * point exists for callers that cannot allocate device memory -- plugins
 * whose host framework owns every byte of HBM, code that must not trigger the
 * device-wide synchronisation of cudaMalloc/cudaFree, and callers without
 * access to any allocator, torch's included.
 *
 * Same arguments, layouts, numerics and validation as ffn_forward (M <= 32,
 * else TFFN_ERR_INVALID_ARG).  The caller passes inputs and outputs; all
 * scratch (control word, ready flags, split-K counters, H, partial sums) lives
 * in one static 16 MiB device array in the library, held by every GPU that
 * loads it until the process exits.  A shape whose scratch does not fit
 * returns TFFN_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on each device fetches the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array and clears its flags and counters
 *     (cudaMemsetAsync) on `stream` before its kernel: calls that overlap on
 *     the GPU (different streams, not ordered) race and corrupt each other.
 *   - It calls no cudaMalloc, cudaFree or allocating routine, and does not use
 *     or need the workspace of the other entry points.
 *   - Its device waits are bounded by TFFN_OPT_WAIT_LIMIT_MS like every other
 *     path.  A wait that ran out of time leaves Y incomplete and records the
 *     error in the array's control block: tffn_check_noalloc() reads it.  The
 *     next call clears the record, so check before calling again.
 */
int ffn_forward_decode_noalloc(const void* X, const void* W1, const void* b1, const void* W2,
                               const void* b2, int act1, int act2, int64_t M, int64_t N, int64_t O,
                               int64_t P, void* Y, struct CUstream_st* stream);

/* Error query of ffn_forward_decode_noalloc: synchronise `stream`, then read
 * and clear the device-side error record in the static scratch array of the
 * current device.  Like that entry point it has no counterpart in the paper;
 * it exists because tffn_check() reads the workspace of the other entry
 * points, which a caller that cannot allocate never has.  Returns TFFN_OK
 * (also when no call ran on this device), TFFN_ERR_TIMEOUT, TFFN_ERR_DEVICE,
 * or TFFN_ERR_CUDA if the synchronisation or the 16-byte read failed; it
 * allocates nothing.  `detail` (nullable, 4 entries) receives {status, wait
 * site, block, info}. */
int tffn_check_noalloc(struct CUstream_st* stream, int32_t* detail);

/* Bytes of workspace a call of this shape needs on the current device
 * (E = 0: ffn_forward or ffn_glu_forward, whichever needs more; E >= 1:
 * moe_ffn_forward with top_k).  Without a usable device the decode part is
 * sized for up to 1024 CTAs. */
size_t tffn_workspace_bytes(int64_t M, int64_t N, int64_t O, int64_t P, int E, int top_k);

/* Use a caller-owned device buffer (>= 256-byte aligned) as the workspace of
 * the current device from the next call on; NULL returns to the
 * library-owned workspace.  The library initialises the buffer's control and
 * flag region on the next call's stream. */
int tffn_set_workspace(void* dev_ptr, size_t bytes);

/* Synchronise `stream`, then read and clear the current device's device-side
 * error record.  Returns TFFN_OK, TFFN_ERR_TIMEOUT or TFFN_ERR_DEVICE (or
 * TFFN_ERR_CUDA if the synchronisation itself failed).  `detail` (nullable,
 * 4 entries) receives {status, wait site, block, info}. */
int tffn_check(struct CUstream_st* stream, int32_t* detail);

/* Static description of a status code. */
const char* tffn_status_string(int status);

/* Tuning and test controls (process-wide):
 *   TFFN_OPT_PATH         0 auto, 1 fused engine, 2 decode stream, 3 engine
 *                         as two launches (layer 1, then layer 2), 4 the
 *                         reduce-add form of "Kernel fusion and tensor
 *                         parallelism", section "Step 1" (each H tile times
 *                         its row of W2 tiles, reduced asynchronously into an
 *                         fp32 Y; results vary in the last bits run to run),
 *                         5 back-to-back (each task walks the hidden tiles of
 *                         one band for one Y tile, H only in shared memory,
 *                         products summed in tensor memory; for small FFNs),
 *                         6 the tensor-core weight stream (up to 256 rows;
 *                         the weights as the MMA's M side); 4 and 5
 *                         apply to ffn_forward only; other values are refused
 *                         (-1, option unchanged)
 *   TFFN_OPT_WAIT_LIMIT_MS  device wait limit in ms (default 4000)
 *   TFFN_OPT_SKIP_FLAG    test fault injection (-1 = off): the engine never
 *                         publishes the ready flag of this GEMM1 tile index,
 *                         and the dense decode stream (ffn_forward up to 32
 *                         rows, and ffn_forward_decode_noalloc) never
 *                         publishes the flags of this 128-column H slice; the
 *                         waiting GEMM2 work then times out and the call
 *                         reports TFFN_ERR_TIMEOUT through tffn_check() (or
 *                         tffn_check_noalloc())
 *   TFFN_OPT_GROUP_M      row bands per raster group of the engine; 0
 *                         (default): 8 when N >= 8192, else 4 (the measured
 *                         optima on GB300)
 *   TFFN_OPT_MOE_ORDER    order of the experts' row segments in the grouped
 *                         layout: 0 expert index, 1 (default) largest row
 *                         count first.  Results are identical either way.
 *   TFFN_OPT_MOE_COMBINE  1 (default): the gate-weighted sum of a token's
 *                         expert outputs is formed in the expert FFN's layer-2
 *                         epilogue by the last of the token's rows to finish
 *                         (when T x ceil(P/256) counters fit the workspace's
 *                         sync region, else as 0); 0: a separate combine
 *                         kernel.  Results are identical either way.
 * Returns the previous value. */
enum {
    TFFN_OPT_PATH = 1,
    TFFN_OPT_WAIT_LIMIT_MS = 2,
    TFFN_OPT_SKIP_FLAG = 3,
    TFFN_OPT_GROUP_M = 4,
    TFFN_OPT_MOE_ORDER = 5,
    TFFN_OPT_MOE_COMBINE = 6
};
int64_t tffn_set_option(int option, int64_t value);

/* Kernels the most recent forward call on this thread launched. */
int tffn_last_launch_count(void);

/* Timing of the dominant kernel (the engine, or the decode stream): while
 * enabled, each forward call records a CUDA event pair around its dominant
 * kernel on the call's stream.  tffn_timing_end synchronises those events and
 * returns the number of timed launches and their summed milliseconds. */
int tffn_timing_begin(void);
int tffn_timing_end(int* launches, double* total_ms);
/* Time only one dominant launch of every `every` (>= 1; default 1) from the
 * next tffn_timing_begin on: an event pair recorded between two kernels
 * serialises them, so sampling keeps most launches back to back.  Returns
 * TFFN_ERR_INVALID_ARG for every < 1. */
int tffn_timing_sample(int every);

/* Host-side view of the engine's task order, for tests (no GPU needed):
 * the task of `ticket` for a fused launch with m_blocks row bands, n1 GEMM1
 * and n2 GEMM2 column tiles and raster groups of group_m bands.  out[0] =
 * layer (0 or 1, -1 past the end), out[1] = row band, out[2] = column tile.
 * Returns the total number of tickets, or -1 if the 32-bit form of the
 * mapping that the kernel runs disagrees with this 64-bit one. */
int64_t tffn_debug_engine_task(int64_t m_blocks, int32_t n1, int32_t n2, int32_t group_m,
                               int64_t ticket, int32_t out[3]);

/* Host-side view of a weight stream's work plan, for tests (no GPU needed).
 * path = 2 (mma.sync stream) or 6 (tcgen05 stream), for M x N x O x P on
 * `sms` SMs, glu = 1 for the gated form.  out = {grid, window mode (0 split
 * layer 1; 1 two-block windows; 2 four-block windows), 64-column hidden
 * blocks, slices of layer 1, slices of layer 2, K chunks per slice of layer 1
 * (window: chunks of the window's K loop), K chunks per slice of layer 2,
 * units of layer 1, units of layer 2, most parts of one slice in layer 1 and
 * in layer 2, bytes of split-K partial sums}.  Returns TFFN_OK,
 * TFFN_ERR_INVALID_ARG for another path or non-positive sizes, or
 * TFFN_ERR_UNSUPPORTED past the stream's 256 rows. */
int tffn_debug_stream_plan(int path, int64_t M, int64_t N, int64_t O, int64_t P, int sms, int glu,
                           int64_t out[12]);

/* Tile sizes of the engine (rows, columns, k-step) and of the decode stream,
 * for tests and tools: out[0..5] = {BM, BN, BK, stages, decode slice width,
 * decode k chunk}. */
void tffn_debug_tiles(int32_t out[6]);

#ifdef __cplusplus
}
#endif
#endif /* TFFN_H */
