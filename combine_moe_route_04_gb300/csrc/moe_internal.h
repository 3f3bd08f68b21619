// moe_internal.h -- host-side declarations shared by the library's
// translation units (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

// Bits ORed into the workspace status word by kernels.
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBounds = 2u;

constexpr int kRowBlock = 128;      // rows per expert block (the expert alignment unit)
constexpr int kChunkTokens = 32;    // tokens per routing histogram chunk (one warp)

inline int64_t max_blocks_of(const moe_shape& s) {
  const int64_t R = static_cast<int64_t>(s.T) * s.k;
  const int64_t touched = R < s.E ? R : s.E;
  return (R + (kRowBlock - 1) * touched) / kRowBlock;
}
inline int64_t max_rows_of(const moe_shape& s) { return kRowBlock * max_blocks_of(s); }
// The GEMMs cut an expert's c rows into ceil(c / kWindowRows) token windows;
// their number over all experts is at most T*k / kWindowRows + min(E, T*k).
constexpr int kWindowRows = 256;
inline int64_t max_windows_of(const moe_shape& s) {
  const int64_t tk = static_cast<int64_t>(s.T) * s.k;
  return tk / kWindowRows + (s.E < tk ? s.E : tk);
}
inline int64_t num_chunks_of(const moe_shape& s) { return (s.T + kChunkTokens - 1) / kChunkTokens; }
// The hand-off counters of one forward: the gate/up tiles stored per token
// window.
inline int64_t forward_counters_of(const moe_shape& s) { return max_windows_of(s); }
// columns of X copied per work item of the row gathers
constexpr int kGatherCols = 1024;
inline int gather_pieces_of(const moe_shape& s) { return (s.H + kGatherCols - 1) / kGatherCols; }

// Byte offsets of everything the workspace holds.
struct WsLayout {
  size_t status;        // uint32 status word (+ padding)
  size_t chunk_counts;  // int32 [E][num_chunks]: per-chunk expert histogram, later chunk bases
  size_t xp;            // bf16 [max_rows][H]: gathered activation rows
  size_t topk_ids, topk_w, counts, off_pad, block_expert, num_blocks, gather_idx, scatter_idx;
  size_t local_rank;    // int32 [T][k]: a forward's in-chunk ranks (routing -> permutation)
  size_t h;             // bf16 [max_rows][I]
  size_t y;             // bf16 [max_rows][H]
  size_t win_done;      // uint32 [forward_counters]: a forward's per-window gate/up tile counts
  size_t total;
};
WsLayout ws_layout(const moe_shape& s);

// Puts the calling thread's previous current device back when an entry point
// returns, if device_ready changed it.
struct DeviceRestore {
  int prev = -1;
  DeviceRestore() = default;
  DeviceRestore(const DeviceRestore&) = delete;
  DeviceRestore& operator=(const DeviceRestore&) = delete;
  ~DeviceRestore() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

// Makes the stream's device current for the launches that follow (recording
// the previous one in `restore`) and checks it (compute capability 10.3);
// fetches the tensor-map encoder on first use.
moe_status device_ready(cudaStream_t st, int* num_sms, DeviceRestore* restore);
// The shape checks every entry point applies (MOE_OK or the error code).
moe_status validate_shape(const moe_shape* s);

inline uint32_t* ws_status(void* ws) { return reinterpret_cast<uint32_t*>(ws); }
// tile-scheduler counters of the two GEMMs, inside the first 256 bytes that
// moe_workspace_init clears (separate 64-byte lines)
inline uint32_t* ws_sched_up(void* ws) { return reinterpret_cast<uint32_t*>(ws) + 16; }
inline uint32_t* ws_sched_down(void* ws) { return reinterpret_cast<uint32_t*>(ws) + 32; }
// the status word as a forward's row gather found it (see the down GEMM's
// per-window wait), in the same cleared 256 bytes
constexpr int kStatusSnapshotIndex = 48;
// the routing's chunk counter (the CTA that brings it to the chunk count scans
// the histograms; the next kernel puts it back to zero) and the mark that scan
// leaves, two words in the same cleared 256 bytes
inline uint32_t* ws_route_counter(void* ws) { return reinterpret_cast<uint32_t*>(ws) + 56; }

// Launch with programmatic stream serialisation (the kernel must call
// pdl_wait() before touching memory its predecessors use).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launchers (asynchronous; return cudaGetLastError()).
// route_counter: a uint32 that is zero between calls (the call leaves it so).
cudaError_t launch_route(const moe_shape& s, const float* logits, int32_t* topk_ids, float* topk_w,
                         int32_t* counts, int32_t* off_pad, int32_t* block_expert, int32_t* num_blocks,
                         int32_t* gather_idx, int32_t* scatter_idx, int32_t* chunk_counts,
                         uint32_t* route_counter, uint32_t* status, cudaStream_t st);

// Inside moe_forward: the routing's first kernel, then one kernel that builds
// the permutation and gathers the rows (Xp[scatter_idx[t, j]] = X[t], each row
// of X read once).  local_rank: [T, k] int32 scratch.  fwd_counters: the
// forward's n_fwd hand-off counters, cleared by the second kernel (which also
// records the status word as the forward found it).
cudaError_t launch_route_gather(const moe_shape& s, const float* logits, const uint16_t* X, int32_t* topk_ids,
                                float* topk_w, int32_t* counts, int32_t* off_pad, int32_t* block_expert,
                                int32_t* num_blocks, int32_t* gather_idx, int32_t* scatter_idx,
                                int32_t* local_rank, int32_t* chunk_counts, uint16_t* Xp, uint32_t* route_counter,
                                uint32_t* fwd_counters, int64_t n_fwd, uint32_t* status, int num_sms,
                                cudaStream_t st);

// Xp[scatter_idx[t, j]] = X[t] for every (t, j), token by token (each row of
// X read once).
cudaError_t launch_scatter_rows(const moe_shape& s, const uint16_t* X, const int32_t* scatter_idx, uint16_t* Xp,
                                uint32_t* status, cudaStream_t st);

struct GemmMaps {
  CUtensorMap a;     // token rows (K-major): Xp [max_rows][H] or h [max_rows][I]; box 128 x 32
  CUtensorMap b0;    // weights, up: W_gate [E*H][I]; down: W_down [E*I][H]; box 32 x 64
  CUtensorMap b1;    // weights, up: W_up   [E*H][I]; down: unused (copy of b0)
  CUtensorMap a64;   // the same token rows, box 64 x 32 (windows of <= 128 rows)
  CUtensorMap a80;   // the same token rows, box 80 x 32 (windows of <= 160 rows)
};

// sched: the kernel's tile counter and its done counter (two uint32 in the
// workspace's first 256 bytes, zero between launches)
// win_done (max_windows_of(s) counters, or nullptr): within one forward the
// gate/up GEMM counts each window's stored tiles there and the down GEMM that
// follows waits per window instead of for the whole previous grid.
cudaError_t launch_gemm_up(const moe_shape& s, const GemmMaps& maps, uint16_t* h, const int32_t* off_pad,
                           const int32_t* counts, uint32_t* status, uint32_t* sched, uint32_t* win_done,
                           int num_sms, cudaStream_t st);
cudaError_t launch_gemm_down(const moe_shape& s, const GemmMaps& maps, uint16_t* Y, const int32_t* off_pad,
                             const int32_t* counts, uint32_t* status, uint32_t* sched, uint32_t* win_done,
                             int num_sms, cudaStream_t st);

cudaError_t launch_combine(const moe_shape& s, const uint16_t* Y, const int32_t* scatter_idx,
                           const float* topk_w, uint16_t* out, uint32_t* status, int num_sms, cudaStream_t st);

// Diagnostic: one thread waits on an mbarrier that nothing arrives on, through
// the library's bounded wait; records kStatusTimeout after kWaitLimitNs.
cudaError_t launch_wait_timeout(uint32_t* status, cudaStream_t st);

// Tensor-map encoding through the driver entry point (no link-time libcuda).
// rows x cols bf16 row-major, box = box_cols (inner) x box_rows; the swizzle
// span equals the box's inner extent in bytes (64 or 128).
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_cols);

}  // namespace moe
