/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts expert layer.
 *
 * The layer, per token t with router logits l[t, :] over E experts:
 *   1. route:   softmax over the E logits, the k largest picked (ties to the
 *               lower expert index, slot j = j-th pick), weights renormalised
 *               over the picks;
 *   2. permute: the T*k routed rows grouped by expert into 128-row blocks
 *               (each expert's group padded to a multiple of 128 rows),
 *               tokens ascending inside an expert;
 *   3. up:      per block of expert e, h = bf16(SiLU(A Wg[e]) * (A Wu[e]));
 *   4. down:    Y = bf16(h Wd[e]);
 *   5. combine: out[t] = bf16(sum_j w[t,j] * Y[row(t,j)]), float32, slot order.
 * Sources: "通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §1 (the serial
 * layer: gate/up GEMM -> SiLU -> down GEMM) and §4 (table of data-flow
 * patterns: "dispatch + GEMM" reorders rows by the route, "GEMM + combine" is
 * the top-k weighted reduction); "通算融合算子（三）：ThunderKittens 多卡编程与
 * 可融合的 GEMM 模板" §4 (grouped GEMM over expert row blocks of 128 rows, 128 =
 * expert alignment unit, expert-major task order).
 *
 * Conventions for every call below:
 *   - all tensor pointers are DEVICE pointers, 16-byte aligned, dense
 *     row-major; bf16 tensors are passed as raw 16-bit patterns (moe_bf16);
 *   - the caller owns every buffer; the library allocates no device memory;
 *   - calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise, except moe_workspace_size,
 *     moe_capacity (host only) and moe_last_device_status (synchronises);
 *   - argument and shape errors are returned before anything is launched;
 *     a failed launch returns MOE_ERR_CUDA; errors found by the kernels
 *     themselves (a bounded wait that ran out, an index out of range) are
 *     recorded in the workspace status word and reported by
 *     moe_last_device_status;
 *   - results are bitwise reproducible run to run (no floating-point atomics);
 *   - the step calls and moe_forward may be recorded into a CUDA graph by
 *     stream capture (they only launch kernels on `stream`; the launches keep
 *     their programmatic-dependent-launch edges); moe_last_device_status
 *     synchronises and is not capturable;
 *   - the device must have compute capability 10.3 (GB300), else MOE_ERR_ARCH;
 *   - a call makes the stream's device current for its launches and puts the
 *     calling thread's previous current device back before it returns.
 *
 * Supported shapes (else MOE_ERR_UNSUPPORTED_SHAPE): 1 <= T <= 2^22,
 * 1 <= E <= 256, 1 <= k <= min(E, 16), 128 <= H <= 32768 and
 * 128 <= I <= 32768 with H % 128 == 0 and I % 128 == 0.
 *
 * Capacity: max_blocks = (T*k + 127*min(E, T*k)) / 128 bounds the number of
 * 128-row blocks of any routing; max_rows = 128 * max_blocks.  Buffers indexed
 * by permuted row (gather_idx, h, Y) hold max_rows rows; block_expert holds
 * max_blocks entries.  Only the first num_blocks (device value) blocks are
 * meaningful; entries past them are left unwritten.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;                 /* raw bfloat16 bits */
typedef struct CUstream_st *moe_stream_t;  /* == cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* NULL pointer or NULL shape */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the supported range */
    MOE_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
    MOE_ERR_ARCH = 4,               /* device is not compute capability 10.3 */
    MOE_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
    MOE_ERR_TIMEOUT = 6,            /* a kernel's bounded wait ran out */
    MOE_ERR_DEVICE_BOUNDS = 7,      /* a kernel met an index out of range */
    MOE_ERR_SCRATCH_LIMIT = 8       /* moe_route_noalloc: shape needs more than its fixed scratch */
} moe_status;

typedef struct {
    int32_t T;  /* tokens */
    int32_t H;  /* hidden size */
    int32_t I;  /* expert intermediate size */
    int32_t E;  /* experts */
    int32_t k;  /* experts per token */
} moe_shape;

/* Human-readable name of a status code (static storage). */
const char *moe_status_string(moe_status s);

/* Host only.  Writes max_blocks and max_rows (see Capacity above). */
moe_status moe_capacity(const moe_shape *shape, int64_t *max_blocks, int64_t *max_rows);

/* Host only.  Bytes of the workspace `ws` that every call below accepts
 * (the largest need, that of moe_forward).  One workspace serves all calls
 * of one shape; calls sharing it must be ordered on one stream. */
moe_status moe_workspace_size(const moe_shape *shape, size_t *bytes);

/* Clears the first 256 bytes of `ws`: the status word, the routing's chunk
 * counter and scan mark, both GEMMs' tile counters and the slot where each
 * forward records the status it started with.  Call once after allocating `ws` (asynchronous,
 * on `stream`); the kernels leave their counters cleared for the next call.
 * On a workspace that was never cleared the routing may scan its histograms
 * early and a GEMM may skip tiles; each reports MOE_ERR_DEVICE_BOUNDS when a
 * counter is out of range, and the next call finds the counters cleared.  (The per-window counts of moe_forward, further
 * on in `ws`, are cleared by every forward itself.) */
moe_status moe_workspace_init(const moe_shape *shape, void *ws, moe_stream_t stream);

/* Synchronises `stream`, returns the error recorded by the kernels since the
 * last call (MOE_OK if none) and clears it. */
moe_status moe_last_device_status(void *ws, moe_stream_t stream);

/* Diagnostic for the kernels' bounded waits: launches one thread that waits
 * on an mbarrier nothing arrives on, through the same bounded wait as every
 * pipeline of the library.  After the wait limit (2 s) the kernel records a
 * timeout in the status word at the start of `ws` (a workspace, or any 16-byte
 * aligned device buffer of at least 4 bytes whose first word is the status
 * word) and returns; the GPU is not faulted.  The next
 * moe_last_device_status(ws) returns MOE_ERR_TIMEOUT.  Asynchronous like the
 * step calls; the stream is busy for about 2 s. */
moe_status moe_check_wait_timeout(void *ws, moe_stream_t stream);

/* Steps 1-2: routing, histogram, padded block table and permutation.
 * Passages: "通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §4, table row
 * "dispatch + GEMM" (the routed rows are reordered by the route before the
 * GEMM); "Lecture 11: Programming Systems for Specialized Hardware" example 4
 * (softmax as exp -> sum -> divide); "通算融合算子（三）：ThunderKittens 多卡编程与
 * 可融合的 GEMM 模板" §4 (128 rows = task block = expert alignment unit).
 *   logits       [T, E]  float32 (finite values)
 *   topk_ids     [T, k]  int32  out: picked experts, slot order
 *   topk_w       [T, k]  float32 out: renormalised weights
 *   counts       [E]     int32  out: rows per expert
 *   off_pad      [E+1]   int32  out: first padded row of each expert, off_pad[E] = 128*num_blocks
 *   block_expert [max_blocks] int32 out: expert of each 128-row block
 *   num_blocks   [1]     int32  out: number of blocks (stays on the device)
 *   gather_idx   [max_rows] int32 out: token of each permuted row, -1 for padding
 *   scatter_idx  [T, k]  int32  out: permuted row of each (token, slot)
 *   ws           workspace (scratch: per-chunk expert histograms; the chunk
 *                counter in its cleared first 256 bytes)
 * Counts, table and permutation are exact; topk_ids are exact for the
 * float32 logits given; topk_w is within a few float32 ulps of the
 * correctly rounded value. */
moe_status moe_route(const moe_shape *shape, const float *logits,
                     int32_t *topk_ids, float *topk_w, int32_t *counts,
                     int32_t *off_pad, int32_t *block_expert, int32_t *num_blocks,
                     int32_t *gather_idx, int32_t *scatter_idx, void *ws,
                     moe_stream_t stream);

/* moe_route without a workspace: the same kernels and the same outputs as
 * moe_route, but the per-chunk expert histograms live in a fixed scratch
 * array that the library places in device memory when it is loaded, so the
 * caller passes only the inputs and outputs and nothing is allocated.  For
 * callers that are not allowed to allocate device memory: a plugin whose host
 * framework owns all device memory and hands it only its inputs and outputs,
 * or a deployment that reserves its memory up front and forbids allocation
 * once running (cudaMalloc may also synchronise the device and stall other
 * streams).  The pages describe no such variant; it has no counterpart there.
 *   - Limit: E * ceil(T/32) <= 262144 (1 MiB of int32 histograms, plus 256
 *     bytes for two counter words; e.g. E=128 with T up to 65536, E=256 with T up to
 *     32768); larger shapes return MOE_ERR_SCRATCH_LIMIT and launch nothing.
 *   - The scratch is one array per device, shared by every call and held
 *     until the process exits.  Calls whose work may overlap on the GPU (on
 *     different streams without ordering) race on it; order them on one
 *     stream.  Every histogram entry a call reads is written earlier in the
 *     same call, and the counter that must start at zero is zero when the
 *     library is loaded and is put back to zero by every call (the scan
 *     mark beside it is cleared at the start of every call), so nothing
 *     needs clearing between calls.
 *   - The first call on a device looks up the scratch address on that device
 *     (a host-side query, no allocation) and caches it.  That lookup may load
 *     the library's module on the device, so make the first call on each
 *     device before capturing any stream into a CUDA graph.
 *   - Kernel-side errors are not reported (there is no status word).
 * Arguments as moe_route, without ws. */
moe_status moe_route_noalloc(const moe_shape *shape, const float *logits,
                             int32_t *topk_ids, float *topk_w, int32_t *counts,
                             int32_t *off_pad, int32_t *block_expert, int32_t *num_blocks,
                             int32_t *gather_idx, int32_t *scatter_idx,
                             moe_stream_t stream);

/* Step 3: grouped gate/up GEMM with the SiLU(gate)*up epilogue.
 * Passages: "通算融合算子（三）：ThunderKittens 多卡编程与可融合的 GEMM 模板" §4
 * (grouped GEMM: each expert's rows multiply that expert's weights, tasks in
 * expert order); "通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §1 (gate/up
 * GEMM followed by SiLU; fused here into the GEMM's epilogue).
 * The GEMM finds each expert's rows from counts and off_pad (rows off_pad[e]
 * .. off_pad[e] + counts[e]) instead of from the block table, and cuts them
 * into windows of at most 256 rows; block_expert and num_blocks are not read.
 *   X          [T, H] bf16 tokens
 *   scatter_idx, counts, off_pad: moe_route's outputs; the call first copies
 *              X[t] to permuted row scatter_idx[t, j] of a workspace buffer
 *              (token by token, so each row of X is read once), then runs
 *              the GEMM over each expert's rows
 *   W_gate [E, H, I] bf16,  W_up [E, H, I] bf16
 *   h          [max_rows, I] bf16 out: h[r] = bf16(silu(g) * u) for every real
 *              row r (gather_idx[r] >= 0); padding rows hold values of no
 *              meaning (never read by the combine)
 *   ws         workspace (scratch: the gathered activation rows; the tile
 *              counter the kernel's clusters draw their tiles from)
 * g and u accumulate in float32 on the tensor cores; SiLU*up is formed in
 * float32 and rounded once to bf16. */
moe_status moe_grouped_gemm_up(const moe_shape *shape, const moe_bf16 *X,
                               const int32_t *scatter_idx, const int32_t *counts,
                               const int32_t *off_pad, const moe_bf16 *W_gate,
                               const moe_bf16 *W_up, moe_bf16 *h, void *ws,
                               moe_stream_t stream);

/* Step 3 on rows already grouped by expert (for callers whose dispatch
 * delivers them that way, as the expert-parallel dispatch of "通算融合算子（一）"
 * §4 does): the same GEMM and epilogue as moe_grouped_gemm_up, without the
 * row gather.
 *   Xp         [max_rows, H] bf16: row r holds the token of permuted row r
 *              (the rows of expert e from off_pad[e], counts[e] of them;
 *              padding rows are not read into any stored result)
 *   counts, off_pad, W_gate, W_up, h: as for moe_grouped_gemm_up
 *   ws         workspace (the tile counter, the status word) */
moe_status moe_grouped_gemm_up_rows(const moe_shape *shape, const moe_bf16 *Xp,
                                    const int32_t *counts, const int32_t *off_pad,
                                    const moe_bf16 *W_gate, const moe_bf16 *W_up,
                                    moe_bf16 *h, void *ws, moe_stream_t stream);

/* Step 4: grouped down GEMM.
 * Passages: "通算融合算子（三）：ThunderKittens 多卡编程与可融合的 GEMM 模板" §4 (the
 * same grouped GEMM); "通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §1 (the
 * down GEMM after SiLU).  Like the gate/up call it takes counts and off_pad in
 * place of the block table.
 *   h      [max_rows, I] bf16 (permuted rows), counts / off_pad from moe_route,
 *   W_down [E, I, H] bf16
 *   Y      [max_rows, H] bf16 out: Y[r] = bf16(h[r] W_down[expert of r]) for
 *          every real row r; padding rows hold values of no meaning */
moe_status moe_grouped_gemm_down(const moe_shape *shape, const moe_bf16 *h,
                                 const int32_t *counts, const int32_t *off_pad,
                                 const moe_bf16 *W_down, moe_bf16 *Y, void *ws,
                                 moe_stream_t stream);

/* Step 5: top-k weighted combine back to token order, without atomics.
 * Passage: "通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §4, table row
 * "GEMM + combine" (the epilogue's top-k weighted reduction).
 *   out[t, c] = bf16(sum_{j<k} topk_w[t,j] * Y[scatter_idx[t,j], c])
 * with a float32 accumulator in slot order, each product and each sum rounded
 * to float32 (no fused multiply-add).
 *   Y [max_rows, H] bf16, scatter_idx [T, k] int32, topk_w [T, k] float32,
 *   out [T, H] bf16; ws: workspace for the status word, or NULL (a row
 *   index outside [0, max_rows) then contributes zero without a report) */
moe_status moe_combine(const moe_shape *shape, const moe_bf16 *Y,
                       const int32_t *scatter_idx, const float *topk_w,
                       moe_bf16 *out, void *ws, moe_stream_t stream);

/* Steps 1-5 on one stream with no host synchronisation in between; all
 * intermediates live in `ws` (see moe_workspace_views).  Passages: those of
 * the five steps above; the per-window hand-off below follows the gate /
 * epilogue hooks of "通算融合算子（三）" §4 (a producer signals a counter per row
 * block, a consumer waits on it) inside one GPU.  Unlike the step
 * calls, which start each kernel after the previous one has completed, the
 * down GEMM here starts on each expert's token window as soon as every
 * gate/up tile of that window is stored (a per-window count kept in `ws`,
 * cleared by the row gather of each forward), so it fills the SMs the gate/up
 * GEMM frees.  The output is bit-identical to the step calls'. */
moe_status moe_forward(const moe_shape *shape, const float *logits, const moe_bf16 *X,
                       const moe_bf16 *W_gate, const moe_bf16 *W_up,
                       const moe_bf16 *W_down, moe_bf16 *out, void *ws,
                       moe_stream_t stream);

/* Device pointers to the intermediates that moe_forward leaves in `ws`
 * (valid after the forward's work on the stream has completed). */
typedef struct {
    int32_t *topk_ids;
    float *topk_w;
    int32_t *counts;
    int32_t *off_pad;
    int32_t *block_expert;
    int32_t *num_blocks;
    int32_t *gather_idx;
    int32_t *scatter_idx;
    moe_bf16 *h;
    moe_bf16 *Y;
    moe_bf16 *Xp;   /* [max_rows, H]: the gathered token rows in expert order */
} moe_views;

moe_status moe_workspace_views(const moe_shape *shape, void *ws, moe_views *views);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
