// moe_route.cu -- routing, expert histogram, 128-row padded block table and
// the gather/scatter permutation, in three small kernels.
//
// What it computes ("通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §4, table
// of data-flow patterns: "dispatch + GEMM" reorders the rows by the route;
// "通算融合算子（三）：ThunderKittens 多卡编程与可融合的 GEMM 模板" §4: rows grouped by
// expert, 128 rows = task block = expert alignment unit; softmax as
// exp -> sum -> divide, "Lecture 11: Programming Systems for Specialized
// Hardware" example 4):
//   per token: softmax over E logits, k largest by logit (ties to the lower
//   index), weights renormalised over the picks;
//   counts[e], off_pad = exclusive scan of ceil(counts/128)*128, block table,
//   row of (t, j) = off_pad[e] + #{t' < t routed to e} (stable by token).
//
// Kernels:
//   1. route_topk_hist: one CTA = one chunk of 32 tokens, one warp per token
//      (warp max / argmax by shuffles); then warp 0 ranks the chunk's T*k
//      entries with __match_any_sync + popc (stable in-chunk rank per expert)
//      and writes the chunk's expert histogram.
//   2. route_scan: one CTA; per expert a warp scans the chunk histograms
//      (chunk bases), then the padded exclusive scan over experts, the block
//      table and the -1 fill of padding rows.
//   3. route_scatter: one thread per (t, j): row = off_pad[e] + chunk base +
//      in-chunk rank; writes scatter_idx and gather_idx.
// Integer atomics are not used, so every output is a pure function of the
// logits.
#include <cfloat>
#include <cstdint>
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxEPerLane = kMaxE / 32;

struct Cand {
  float v;   // logit
  int e;     // expert index
  float x;   // exp(logit - max)
};

// exp(v - m) for float32 v <= m: the difference is split exactly into
// d_hi + d_lo (2Sum) and exp(d_hi + d_lo) ~= exp(d_hi) * (1 + d_lo), so the
// result carries expf's error only, not the rounding of v - m (which grows
// with |v - m|).
__device__ __forceinline__ float exp_diff(float v, float m) {
  const float d_hi = v - m;
  const float bb = d_hi - v;
  const float d_lo = (v - (d_hi - bb)) + (-m - bb);
  const float e = expf(d_hi);
  return fmaf(e, d_lo, e);
}

__device__ __forceinline__ bool better(float va, int ea, float vb, int eb) {
  return va > vb || (va == vb && ea < eb);
}

__global__ void __launch_bounds__(1024) route_topk_hist_kernel(const float* __restrict__ logits, int T, int E,
                                                               int k, int nch, int32_t* __restrict__ topk_ids,
                                                               float* __restrict__ topk_w,
                                                               int32_t* __restrict__ local_rank,
                                                               int32_t* __restrict__ chunk_counts) {
  __shared__ int32_t s_ids[kChunkTokens * kMaxK];
  __shared__ int32_t s_cnt[kMaxE];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int chunk = blockIdx.x;
  const int t0 = chunk * kChunkTokens;
  const int ntok = min(kChunkTokens, T - t0);

  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;

  if (warp < ntok) {
    const int t = t0 + warp;
    const float* row = logits + static_cast<int64_t>(t) * E;
    float v[kMaxEPerLane];
    float x[kMaxEPerLane];
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < kMaxEPerLane; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? __ldg(row + e) : -FLT_MAX;
      if (e < E) m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
#pragma unroll
    for (int i = 0; i < kMaxEPerLane; ++i) x[i] = (lane + 32 * i < E) ? exp_diff(v[i], m) : 0.0f;

    uint32_t taken = 0;  // bit i: element i of this lane already picked
    int my_id = 0;
    float my_x = 0.0f;
    for (int j = 0; j < k; ++j) {
      // best unpicked element of this lane (ascending index: strict > keeps the lower)
      Cand c{-INFINITY, 0x7fffffff, 0.0f};
#pragma unroll
      for (int i = 0; i < kMaxEPerLane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && better(v[i], e, c.v, c.e)) c = Cand{v[i], e, x[i]};
      }
      // warp argmax, ties to the lower index
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, c.v, o);
        const int oe = __shfl_xor_sync(0xffffffffu, c.e, o);
        const float ox = __shfl_xor_sync(0xffffffffu, c.x, o);
        if (better(ov, oe, c.v, c.e)) c = Cand{ov, oe, ox};
      }
      if ((c.e & 31) == lane) taken |= 1u << (c.e >> 5);
      if (lane == j) {
        my_id = c.e;
        my_x = c.x;
      }
    }
    // renormalise over the picks: w_j = x_j / sum_{j' in slot order} x_j'
    // (the softmax denominator cancels).  Slots hold non-increasing x, so
    // Fast2Sum keeps the rounding error of each addition.
    float S = 0.0f, comp = 0.0f;
    for (int j = 0; j < k; ++j) {
      const float y = __shfl_sync(0xffffffffu, my_x, j);
      const float t = S + y;
      comp += (S - t) + y;
      S = t;
    }
    S += comp;
    if (lane < k) {
      topk_ids[static_cast<int64_t>(t) * k + lane] = my_id;
      topk_w[static_cast<int64_t>(t) * k + lane] = my_x / S;
      s_ids[warp * k + lane] = my_id;
    }
  }
  __syncthreads();

  if (warp == 0) {
    // stable rank of every (t, j) of the chunk among the chunk's entries of
    // the same expert, entries in (t, j) order
    const int n = ntok * k;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      const bool act = i < n;
      const int key = act ? s_ids[i] : -1 - lane;
      const uint32_t peers = __match_any_sync(0xffffffffu, key);
      int r = 0;
      if (act) r = s_cnt[key] + __popc(peers & lt_mask);
      __syncwarp();
      if (act && (__ffs(peers) - 1) == lane) s_cnt[key] += __popc(peers);
      __syncwarp();
      if (act) local_rank[static_cast<int64_t>(t0) * k + i] = r;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[static_cast<int64_t>(e) * nch + chunk] = s_cnt[e];
}

__global__ void __launch_bounds__(1024) route_scan_kernel(int E, int nch, int64_t max_blocks,
                                                          int32_t* __restrict__ chunk_counts,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ off_pad,
                                                          int32_t* __restrict__ block_expert,
                                                          int32_t* __restrict__ num_blocks,
                                                          int32_t* __restrict__ gather_idx,
                                                          uint32_t* __restrict__ status) {
  __shared__ int32_t s_cnt[kMaxE];
  __shared__ int32_t s_off[kMaxE + 1];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;

  // per expert: exclusive scan of the chunk histograms -> chunk bases
  for (int e = warp; e < E; e += nwarps) {
    int32_t* cc = chunk_counts + static_cast<int64_t>(e) * nch;
    int running = 0;
    for (int c0 = 0; c0 < nch; c0 += 32) {
      const int c = c0 + lane;
      const int v = (c < nch) ? cc[c] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (c < nch) cc[c] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s_cnt[e] = running;
      counts[e] = running;
    }
  }
  __syncthreads();

  // exclusive scan over experts of the 128-padded counts
  if (warp == 0) {
    constexpr int per = kMaxE / 32;
    int local[per];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      local[i] = (e < E) ? (s_cnt[e] + kRowBlock - 1) / kRowBlock * kRowBlock : 0;
      sum += local[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) s_off[e] = run;
      run += local[i];
    }
    if (lane == 31) s_off[E] = incl;
  }
  __syncthreads();

  const int total_rows = s_off[E];
  int nb = total_rows / kRowBlock;
  if (nb > max_blocks) {  // impossible for valid expert ids; keep every later index in range
    if (threadIdx.x == 0) record_status(status, kStatusBounds);
    nb = static_cast<int>(max_blocks);
  }
  for (int e = threadIdx.x; e <= E; e += blockDim.x) off_pad[e] = s_off[e];
  if (threadIdx.x == 0) *num_blocks = nb;

  // block table: expert whose padded range holds row 128*b
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    const int row = b * kRowBlock;
    int lo = 0, hi = E - 1;  // smallest e with s_off[e+1] > row
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid + 1] > row) hi = mid; else lo = mid + 1;
    }
    block_expert[b] = lo;
  }
  // padding rows of every expert
  for (int e = warp; e < E; e += nwarps) {
    const int end = min(s_off[e + 1], nb * kRowBlock);
    for (int r = s_off[e] + s_cnt[e] + lane; r < end; r += 32) gather_idx[r] = -1;
  }
}

__global__ void route_scatter_kernel(int T, int E, int k, int nch, int64_t max_rows,
                                     const int32_t* __restrict__ topk_ids,
                                     const int32_t* __restrict__ off_pad,
                                     const int32_t* __restrict__ chunk_base,
                                     int32_t* __restrict__ scatter_idx,  // in: in-chunk rank, out: row
                                     int32_t* __restrict__ gather_idx, uint32_t* __restrict__ status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(T) * k) return;
  const int t = static_cast<int>(i / k);
  const int e = topk_ids[i];
  if (e < 0 || e >= E) {
    record_status(status, kStatusBounds);
    return;
  }
  const int chunk = t / kChunkTokens;
  const int64_t row =
      static_cast<int64_t>(off_pad[e]) + chunk_base[static_cast<int64_t>(e) * nch + chunk] + scatter_idx[i];
  if (row < 0 || row >= max_rows) {
    record_status(status, kStatusBounds);
    return;
  }
  scatter_idx[i] = static_cast<int32_t>(row);
  gather_idx[row] = t;
}

}  // namespace

cudaError_t launch_route(const moe_shape& s, const float* logits, int32_t* topk_ids, float* topk_w,
                         int32_t* counts, int32_t* off_pad, int32_t* block_expert, int32_t* num_blocks,
                         int32_t* gather_idx, int32_t* scatter_idx, int32_t* chunk_counts, uint32_t* status,
                         cudaStream_t st) {
  const int nch = static_cast<int>(num_chunks_of(s));
  route_topk_hist_kernel<<<nch, 1024, 0, st>>>(logits, s.T, s.E, s.k, nch, topk_ids, topk_w, scatter_idx,
                                                chunk_counts);
  route_scan_kernel<<<1, 1024, 0, st>>>(s.E, nch, max_blocks_of(s), chunk_counts, counts, off_pad, block_expert,
                                        num_blocks, gather_idx, status);
  const int64_t n = static_cast<int64_t>(s.T) * s.k;
  const int threads = 256;
  route_scatter_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, st>>>(
      s.T, s.E, s.k, nch, max_rows_of(s), topk_ids, off_pad, chunk_counts, scatter_idx, gather_idx, status);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------
// moe_route_noalloc: moe_route for callers that may not allocate device
// memory (for instance a plugin whose host framework owns all device memory
// and only hands it input and output buffers, or a deployment that reserves
// its memory up front and forbids allocation once running).  The only scratch
// the routing kernels need -- the per-chunk expert histograms, later the
// chunk bases -- lives in this fixed array instead of a caller workspace.  It
// is placed in device memory when the library's module is loaded on a device
// and stays there until the process exits.
namespace moe {
namespace {

constexpr int64_t kNoAllocScratchInts = int64_t(1) << 18;  // 1 MiB of int32

__device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

int32_t* g_route_scratch_addr[64] = {};
std::mutex g_route_scratch_mu;

// Device address of g_route_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int32_t* route_scratch_on_device(int dev) {
  std::lock_guard<std::mutex> lock(g_route_scratch_mu);
  if (g_route_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_route_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  return g_route_scratch_addr[dev];
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(const moe_shape* shape, const float* logits, int32_t* topk_ids,
                                        float* topk_w, int32_t* counts, int32_t* off_pad, int32_t* block_expert,
                                        int32_t* num_blocks, int32_t* gather_idx, int32_t* scatter_idx,
                                        moe_stream_t stream) {
  using namespace moe;
  moe_status st = validate_shape(shape);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {logits, topk_ids, topk_w, counts, off_pad, block_expert, num_blocks, gather_idx,
                        scatter_idx};
  for (const void* p : ptrs) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return MOE_ERR_MISALIGNED;
  }
  if (static_cast<int64_t>(shape->E) * num_chunks_of(*shape) > kNoAllocScratchInts) return MOE_ERR_SCRATCH_LIMIT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = device_ready(s, nullptr);  // makes the stream's device current
  if (st != MOE_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  int32_t* scratch = route_scratch_on_device(dev);
  if (scratch == nullptr) return MOE_ERR_CUDA;
  // Every chunk-histogram entry the scan and scatter read is written by the
  // first kernel of this call, so stale contents need no clearing.
  const cudaError_t e = launch_route(*shape, logits, topk_ids, topk_w, counts, off_pad, block_expert, num_blocks,
                                     gather_idx, scatter_idx, scratch, /*status=*/nullptr, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
