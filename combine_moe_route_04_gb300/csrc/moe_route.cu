// moe_route.cu -- routing, expert histogram, 128-row padded block table and
// the gather/scatter permutation, in two small kernels.
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
//   1. route_topk_hist: one CTA = one chunk of 32 tokens, one warp per token;
//      each lane sorts its few packed (logit, index) keys, then k rounds of a
//      warp max over the lanes' leading keys (two 32-bit warp reductions: the
//      logit word, then the index word among the tied lanes); each
//      pick sets its token's bit in a per-expert 32-bit mask (shared-memory
//      OR), so an entry's stable in-chunk rank is the popcount of its
//      expert's mask below its token and the chunk's count the whole
//      popcount.  Each CTA then counts its chunk in on a counter; the CTA
//      that counts the last chunk in scans every expert's chunk histogram
//      (the chunk bases) and writes the experts' row counts.
//   2. route_scatter: every CTA scans the padded counts (off_pad) in shared
//      memory; one thread per (t, j) writes row = off_pad[e] + chunk base +
//      in-chunk rank to scatter_idx and gather_idx; the block table and the
//      padding rows' -1 are spread over all threads.
// The only atomics are those shared-memory ORs, whose result does not depend
// on their order, so every output is a pure function of the logits.
#include <cfloat>
#include <cstdint>
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kMaxE = 256;
constexpr int kTopkThreads = 32 * kChunkTokens;              // one warp per token of the chunk

// route_counter[0]: kernel 1's chunk arrivals (zero at the start of a call);
// route_counter[1]: the mark kernel 1's scanning CTA leaves once the chunk
// bases and counts are written (cleared at the start of every call).
__host__ __device__ constexpr uint32_t scan_mark(int nch) { return 0x5CA40000u ^ static_cast<uint32_t>(nch); }

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

// Sort key of (logit, expert): the logit's bits mapped to an unsigned order
// (after -0 -> +0, so the two zeros tie as they compare equal) in the high
// word and 0xFFFF - e in the low word: a larger key is a larger logit, or an
// equal logit with a lower index.  0 is below every real key.
__device__ __forceinline__ uint64_t pick_key(float v, int e) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(0xFFFF - e);
}
__device__ __forceinline__ float key_logit(uint64_t key) {
  const uint32_t ord = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
__device__ __forceinline__ int key_expert(uint64_t key) { return 0xFFFF - static_cast<int>(key & 0xFFFFu); }

// Exclusive scan across the warp of one value per lane; returns the lane's
// exclusive prefix and sets `total` to the warp's sum.
__device__ __forceinline__ int warp_exclusive_scan(int v, int lane, int& total) {
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - v;
}

// One warp: exclusive scans of the chunk histograms of experts ea and eb
// (eb >= E: none) into chunk bases, in place, and their total row counts.
// Both experts' loads are issued before either is scanned, and only the
// 32-chunk batches that exist are scanned.  The histograms were written by
// other CTAs, so they are read through L2 (__ldcg).
__device__ __forceinline__ void scan_expert_pair(int ea, int eb, int E, int nch, int lane,
                                                 int32_t* __restrict__ chunk_counts, int32_t* __restrict__ counts) {
  constexpr int U = 4;  // 32-chunk batches per expert loaded before any is scanned
  int32_t* ca = chunk_counts + static_cast<int64_t>(ea) * nch;
  int32_t* cb = chunk_counts + static_cast<int64_t>(eb < E ? eb : ea) * nch;
  const bool has_b = eb < E;
  int run_a = 0, run_b = 0;
  for (int c0 = 0; c0 < nch; c0 += 32 * U) {
    int va[U], vb[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 32 * u + lane;
      va[u] = (c < nch) ? __ldcg(ca + c) : 0;
      vb[u] = (has_b && c < nch) ? __ldcg(cb + c) : 0;
    }
    const int nb = min(U, (nch - c0 + 31) / 32);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u < nb) {
        const int c = c0 + 32 * u + lane;
        int ta, tb;
        const int xa = warp_exclusive_scan(va[u], lane, ta);
        const int xb = warp_exclusive_scan(vb[u], lane, tb);
        if (c < nch) {
          ca[c] = run_a + xa;
          if (has_b) cb[c] = run_b + xb;
        }
        run_a += ta;
        run_b += tb;
      }
    }
  }
  if (lane == 0) {
    counts[ea] = run_a;
    if (has_b) counts[eb] = run_b;
  }
}

// Kernel 1: one CTA per chunk of 32 tokens, one warp per token: the k best
// experts (k rounds of a warp-wide max over the keys, the winner removed
// each round; slot j = j-th round) and the renormalised weights; then the
// chunk's expert histogram and each entry's stable in-chunk rank from the
// per-expert token masks.  The CTA that finishes the last chunk (the one
// whose arrival on route_counter, zero at the start of the call, returns
// nch - 1) then turns every expert's chunk histogram into chunk bases and
// writes counts; route_scatter puts the counter back to zero.
// EPL = logits per lane (E <= 32 * EPL).
template <int EPL>
__global__ void __launch_bounds__(kTopkThreads) route_topk_hist_kernel(
    const float* __restrict__ logits, int T, int E, int k, int nch, int32_t* __restrict__ topk_ids,
    float* __restrict__ topk_w, int32_t* __restrict__ local_rank, int32_t* __restrict__ chunk_counts,
    int32_t* __restrict__ counts, uint32_t* __restrict__ route_counter, uint32_t* __restrict__ status) {
  __shared__ uint32_t s_mask[kMaxE];  // bit w: token w of the chunk picked expert e
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int chunk = blockIdx.x;
  const int t0 = chunk * kChunkTokens;
  const int ntok = min(kChunkTokens, T - t0);

  for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0u;
  __syncthreads();
  pdl_wait();  // inputs and outputs may be in use by the previous kernel until here
  // the next kernel's CTAs may launch only now: launched earlier, they would
  // wait on SMs the previous kernel (a forward's combine) still needs
  pdl_launch_dependents();
  // no scan has happened in this call yet (thread 0 of CTA 0 clears the mark
  // before its own arrival, so before the scanning CTA can set it)
  if (chunk == 0 && threadIdx.x == 0) route_counter[1] = 0u;

  int my_e = 0;
  if (warp < ntok) {
    const int t = t0 + warp;
    const float* row = logits + static_cast<int64_t>(t) * E;
    uint64_t key[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      key[i] = (e < E) ? pick_key(__ldg(row + e), e) : 0ull;
    }
    // this lane's keys in descending order (a small exchange network)
#pragma unroll
    for (int a = 0; a < EPL - 1; ++a) {
#pragma unroll
      for (int b = EPL - 1; b > a; --b) {
        const uint64_t x = key[b - 1], y = key[b];
        key[b - 1] = x > y ? x : y;
        key[b] = x > y ? y : x;
      }
    }
    // round j: the warp's largest leading key is pick j; its lane pops it
    // (keys are unique, so exactly one lane holds it)
    uint64_t my_key = 0;
    for (int j = 0; j < k; ++j) {
      const uint32_t hi = static_cast<uint32_t>(key[0] >> 32);
      const uint32_t lo = static_cast<uint32_t>(key[0]);
      const uint32_t best_hi = __reduce_max_sync(0xffffffffu, hi);
      const uint32_t best_lo = __reduce_max_sync(0xffffffffu, hi == best_hi ? lo : 0u);
      const uint64_t best = (static_cast<uint64_t>(best_hi) << 32) | best_lo;
      if (key[0] == best) {
#pragma unroll
        for (int i = 0; i < EPL - 1; ++i) key[i] = key[i + 1];
        key[EPL - 1] = 0ull;
      }
      if (lane == j) my_key = best;
    }
    // the first pick is the row maximum
    const float m = key_logit(__shfl_sync(0xffffffffu, my_key, 0));
    my_e = key_expert(my_key);
    const float my_x = (lane < k) ? exp_diff(key_logit(my_key), m) : 0.0f;
    // w_j = x_j / sum_{j' in slot order} x_j' (the softmax denominator
    // cancels); slots hold non-increasing x, so Fast2Sum keeps the rounding
    // error of each addition
    float S = 0.0f, comp = 0.0f;
    for (int j = 0; j < k; ++j) {
      const float y = __shfl_sync(0xffffffffu, my_x, j);
      const float tt = S + y;
      comp += (S - tt) + y;
      S = tt;
    }
    S += comp;
    if (lane < k) {
      topk_ids[static_cast<int64_t>(t) * k + lane] = my_e;
      topk_w[static_cast<int64_t>(t) * k + lane] = my_x / S;
      atomicOr(&s_mask[my_e], 1u << warp);  // a token picks an expert at most once
    }
  }
  __syncthreads();
  // stable rank of (t, j) among the chunk's entries of its expert, entries in
  // (t, j) order = the chunk's earlier tokens that picked the same expert
  if (warp < ntok && lane < k)
    local_rank[static_cast<int64_t>(t0 + warp) * k + lane] = __popc(s_mask[my_e] & ((1u << warp) - 1u));
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<int64_t>(e) * nch + chunk] = __popc(s_mask[e]);

  // count this chunk in (its histogram made visible first); the CTA that
  // counts the last one in scans all histograms.  A count past nch means the
  // counter was not zero at the start (a workspace never cleared).
  __syncthreads();
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();  // release: the CTA's histogram (ordered by the barrier) before the arrival
    const uint32_t ticket = atomicAdd(route_counter, 1u);
    if (ticket >= static_cast<uint32_t>(nch)) record_status(status, kStatusBounds);
    s_last = ticket == static_cast<uint32_t>(nch - 1) ? 1 : 0;
    if (s_last) fence_acq_rel_gpu();  // acquire: every other CTA's histogram
  }
  __syncthreads();
  if (!s_last) return;
  constexpr int kWarps = kTopkThreads / 32;
  for (int e = warp; e < E; e += 2 * kWarps) scan_expert_pair(e, e + kWarps, E, nch, lane, chunk_counts, counts);
  // the bases and counts are written: the next kernel may use them
  if (threadIdx.x == 0) route_counter[1] = scan_mark(nch);
}

// The part of the permutation every permute kernel shares, run by every CTA
// (all threads): off_pad (exclusive scan of the 128-padded counts) into
// shared memory; CTA 0 writes off_pad and num_blocks; the block table and
// the padding rows' gather index -1 spread over all threads.  Also resets
// the first kernel's chunk counter, and inside moe_forward clears the
// forward's hand-off counters and records the status word the forward
// started with.  If kernel 1 left no scan mark (its counter was not zero at
// the start, so no CTA scanned), counts are not this call's: the call
// reports MOE_ERR_DEVICE_BOUNDS and routes every expert empty (CTA 0 writes
// zero counts), so nothing is indexed from stale values.  Returns the number
// of 128-row blocks.
__device__ __forceinline__ int permute_common(int E, int nch, int64_t max_count, int64_t max_blocks,
                                              int32_t* __restrict__ counts,
                                              int32_t* s_off, int32_t* s_cnt, int32_t* s_warp,
                                              int32_t* __restrict__ gather_idx, int32_t* __restrict__ off_pad,
                                              int32_t* __restrict__ block_expert, int32_t* __restrict__ num_blocks,
                                              uint32_t* __restrict__ route_counter,
                                              uint32_t* __restrict__ fwd_counters, int64_t n_fwd,
                                              uint32_t* __restrict__ status) {
  const int tid = threadIdx.x;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // kernel 1 has completed: its chunk counter goes back to zero for the next
  // call (also after a call that found it dirty)
  if (gtid == 0) *route_counter = 0u;
  // inside moe_forward: the forward's hand-off counters start from zero (the
  // previous forward's kernels that used them have completed), and the status
  // word is recorded as this forward found it (a hand-off wait gives up only
  // on an error raised after this point)
  if (fwd_counters != nullptr) {
    for (int64_t i = gtid; i < n_fwd; i += nthreads) fwd_counters[i] = 0u;
    if (gtid == 0 && status != nullptr) status[kStatusSnapshotIndex] = *reinterpret_cast<volatile uint32_t*>(status);
  }
  const int lane = tid & 31, warp = tid >> 5;
  const bool scanned = __ldcg(route_counter + 1) == scan_mark(nch);
  if (!scanned && gtid == 0) record_status(status, kStatusBounds);
  // block-wide exclusive scan of padded counts (E <= 256 = blockDim.x)
  int c = 0;
  if (tid < E && scanned) {
    c = __ldcg(counts + tid);
    if (c < 0 || c > max_count) {  // impossible for a count this call scanned
      record_status(status, kStatusBounds);
      c = 0;
    }
  }
  if (tid < E) s_cnt[tid] = c;
  if (!scanned && blockIdx.x == 0 && tid < E) counts[tid] = 0;
  const int padded = (c + kRowBlock - 1) / kRowBlock * kRowBlock;
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_warp[w];
  if (tid < E) s_off[tid] = wbase + incl - padded;
  if (tid == E - 1) s_off[E] = wbase + incl;
  __syncthreads();

  int nb = s_off[E] / kRowBlock;
  if (nb > max_blocks) {  // impossible for valid expert ids; keep every later index in range
    if (gtid == 0) record_status(status, kStatusBounds);
    nb = static_cast<int>(max_blocks);
  }
  if (blockIdx.x == 0) {
    for (int e = tid; e <= E; e += blockDim.x) off_pad[e] = s_off[e];
    if (tid == 0) *num_blocks = nb;
  }
  // block table: the expert whose padded range holds row 128*b
  for (int64_t b = gtid; b < nb; b += nthreads) {
    const int row = static_cast<int>(b) * kRowBlock;
    int lo = 0, hi = E - 1;  // smallest e with s_off[e+1] > row
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid + 1] > row) hi = mid; else lo = mid + 1;
    }
    block_expert[b] = lo;
  }
  // padding rows of every expert: (e, p) -> row off_pad[e] + counts[e] + p
  for (int64_t g = gtid; g < static_cast<int64_t>(E) * kRowBlock; g += nthreads) {
    const int e = static_cast<int>(g / kRowBlock);
    const int64_t row = static_cast<int64_t>(s_off[e]) + s_cnt[e] + (g % kRowBlock);
    if (row >= 0 && row < s_off[e + 1] && row < static_cast<int64_t>(nb) * kRowBlock) gather_idx[row] = -1;
  }
  return nb;
}

// The permuted row of entry (t, j) picking expert e: the expert's first
// padded row + the rows of earlier chunks + the rank inside the chunk; -1
// (and a recorded error) if out of range.
__device__ __forceinline__ int64_t entry_row(int t, int e, int E, int nch, const int32_t* s_off,
                                             const int32_t* __restrict__ chunk_base, int32_t rank, int64_t max_rows,
                                             uint32_t* status) {
  if (e < 0 || e >= E) {
    record_status(status, kStatusBounds);
    return -1;
  }
  const int64_t row = static_cast<int64_t>(s_off[e]) + __ldg(chunk_base + static_cast<int64_t>(e) * nch + t / kChunkTokens) +
                      rank;
  if (row < 0 || row >= max_rows) {
    record_status(status, kStatusBounds);
    return -1;
  }
  return row;
}

// Kernel 2 (the step call moe_route): the shared part, then one thread per
// (t, j) writes its permuted row to scatter_idx (which held its in-chunk
// rank) and gather_idx.
__global__ void __launch_bounds__(256) route_scatter_kernel(int T, int E, int k, int nch, int64_t max_blocks,
                                                            const int32_t* __restrict__ topk_ids,
                                                            int32_t* __restrict__ counts,
                                                            const int32_t* __restrict__ chunk_base,
                                                            int32_t* __restrict__ scatter_idx,  // in: rank, out: row
                                                            int32_t* __restrict__ gather_idx,
                                                            int32_t* __restrict__ off_pad,
                                                            int32_t* __restrict__ block_expert,
                                                            int32_t* __restrict__ num_blocks,
                                                            uint32_t* __restrict__ route_counter,
                                                            uint32_t* __restrict__ status) {
  __shared__ int32_t s_off[kMaxE + 1];
  __shared__ int32_t s_cnt[kMaxE];
  __shared__ int32_t s_warp[8];
  pdl_launch_dependents();
  pdl_wait();
  permute_common(E, nch, static_cast<int64_t>(T) * k, max_blocks, counts, s_off, s_cnt, s_warp, gather_idx, off_pad,
                 block_expert, num_blocks, route_counter, nullptr, 0, status);
  const int64_t max_rows = max_blocks * kRowBlock;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = gtid; i < static_cast<int64_t>(T) * k; i += nthreads) {
    const int t = static_cast<int>(i / k);
    const int64_t row = entry_row(t, topk_ids[i], E, nch, s_off, chunk_base, scatter_idx[i], max_rows, status);
    if (row < 0) continue;
    scatter_idx[i] = static_cast<int32_t>(row);
    gather_idx[row] = t;
  }
}

// Inside moe_forward, kernel 2 and the row gather in one: the shared part,
// then one warp per (token, piece_cols columns of X; 1024, or fewer when
// there are few tokens): lanes j < k find the rows of
// the token's k entries (the first piece's warp writes scatter_idx and
// gather_idx), and the warp copies that piece of X[t] to each of them, so
// each row of X is read once.  The in-chunk ranks come in a separate buffer
// (local_rank), so no warp overwrites what another still reads.
__global__ void __launch_bounds__(256) permute_gather_kernel(int T, int H, int E, int k, int nch,
                                                             int64_t max_blocks,
                                                             const int32_t* __restrict__ topk_ids,
                                                             const int32_t* __restrict__ local_rank,
                                                             int32_t* __restrict__ counts,
                                                             const int32_t* __restrict__ chunk_base,
                                                             const uint16_t* __restrict__ X,
                                                             uint16_t* __restrict__ Xp,
                                                             int32_t* __restrict__ scatter_idx,
                                                             int32_t* __restrict__ gather_idx,
                                                             int32_t* __restrict__ off_pad,
                                                             int32_t* __restrict__ block_expert,
                                                             int32_t* __restrict__ num_blocks,
                                                             uint32_t* __restrict__ route_counter,
                                                             uint32_t* __restrict__ fwd_counters, int64_t n_fwd,
                                                             int piece_cols, int late_trigger,
                                                             uint32_t* __restrict__ status) {
  __shared__ int32_t s_off[kMaxE + 1];
  __shared__ int32_t s_cnt[kMaxE];
  __shared__ int32_t s_warp[8];
  // The gate/up GEMM's CTAs (one per SM, holding most of its registers) may
  // launch once every CTA here has let them.  With a large gather that is
  // only after this kernel's wait, so they do not take the SMs' registers
  // from the gather's CTAs early; with a small one, at once, so that their
  // prologue runs under this kernel.
  if (!late_trigger) pdl_launch_dependents();
  pdl_wait();
  if (late_trigger) pdl_launch_dependents();
  permute_common(E, nch, static_cast<int64_t>(T) * k, max_blocks, counts, s_off, s_cnt, s_warp, gather_idx, off_pad,
                 block_expert, num_blocks, route_counter, fwd_counters, n_fwd, status);
  const int64_t max_rows = max_blocks * kRowBlock;
  const int CH = piece_cols;  // columns per work item: 16 bytes x (piece_cols / 256) per lane
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int npiece = (H + CH - 1) / CH;
  const int64_t items = static_cast<int64_t>(T) * npiece;
  for (int64_t item = warp0; item < items; item += nwarps) {
    const int t = static_cast<int>(item / npiece);
    const int piece = static_cast<int>(item % npiece);
    const int c0 = piece * CH;
    int my_row = -1;  // lane j < k: row of (t, j)
    if (lane < k) {
      const int64_t i = static_cast<int64_t>(t) * k + lane;
      const int64_t row = entry_row(t, __ldg(topk_ids + i), E, nch, s_off, chunk_base, __ldg(local_rank + i),
                                    max_rows, status);
      if (row >= 0) {
        my_row = static_cast<int>(row);
        if (piece == 0) {
          scatter_idx[i] = my_row;
          gather_idx[row] = t;
        }
      }
    }
    const int nv = min(CH, H - c0) / 8;  // 16-byte vectors in this piece (H % 128 == 0)
    const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(t) * H + c0);
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = lane + 32 * u;
      if (idx < nv) v[u] = __ldg(src + idx);
    }
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      if (row < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(Xp + static_cast<int64_t>(row) * H + c0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = lane + 32 * u;
        if (idx < nv) dst[idx] = v[u];
      }
    }
  }
}

}  // namespace

namespace {

cudaError_t launch_route_topk(const moe_shape& s, const float* logits, int32_t* topk_ids, float* topk_w,
                              int32_t* local_rank, int32_t* chunk_counts, int32_t* counts, uint32_t* route_counter,
                              uint32_t* status, cudaStream_t st) {
  const int nch = static_cast<int>(num_chunks_of(s));
  const int epl = (s.E + 31) / 32;
  auto k1 = epl <= 1 ? route_topk_hist_kernel<1>
          : epl <= 2 ? route_topk_hist_kernel<2>
          : epl <= 4 ? route_topk_hist_kernel<4>
                     : route_topk_hist_kernel<8>;
  return launch_pdl(k1, dim3(nch), dim3(kTopkThreads), 0, st, logits, s.T, s.E, s.k, nch, topk_ids, topk_w,
                    local_rank, chunk_counts, counts, route_counter, status);
}

}  // namespace

cudaError_t launch_route(const moe_shape& s, const float* logits, int32_t* topk_ids, float* topk_w,
                         int32_t* counts, int32_t* off_pad, int32_t* block_expert, int32_t* num_blocks,
                         int32_t* gather_idx, int32_t* scatter_idx, int32_t* chunk_counts,
                         uint32_t* route_counter, uint32_t* status, cudaStream_t st) {
  const int nch = static_cast<int>(num_chunks_of(s));
  // kernel 1 leaves each entry's in-chunk rank in scatter_idx; kernel 2
  // replaces it by the entry's row
  cudaError_t err = launch_route_topk(s, logits, topk_ids, topk_w, scatter_idx, chunk_counts, counts,
                                      route_counter, status, st);
  if (err != cudaSuccess) return err;
  const int64_t n = static_cast<int64_t>(s.T) * s.k;
  const int64_t work = n > static_cast<int64_t>(s.E) * kRowBlock ? n : static_cast<int64_t>(s.E) * kRowBlock;
  int64_t blocks = (work + 255) / 256;
  if (blocks > 1184) blocks = 1184;
  err = launch_pdl(route_scatter_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, s.T, s.E, s.k, nch,
                   static_cast<int64_t>(max_blocks_of(s)), static_cast<const int32_t*>(topk_ids),
                   counts, static_cast<const int32_t*>(chunk_counts), scatter_idx,
                   gather_idx, off_pad, block_expert, num_blocks, route_counter, status);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_route_gather(const moe_shape& s, const float* logits, const uint16_t* X, int32_t* topk_ids,
                                float* topk_w, int32_t* counts, int32_t* off_pad, int32_t* block_expert,
                                int32_t* num_blocks, int32_t* gather_idx, int32_t* scatter_idx,
                                int32_t* local_rank, int32_t* chunk_counts, uint16_t* Xp, uint32_t* route_counter,
                                uint32_t* fwd_counters, int64_t n_fwd, uint32_t* status, int num_sms,
                                cudaStream_t st) {
  const int nch = static_cast<int>(num_chunks_of(s));
  cudaError_t err = launch_route_topk(s, logits, topk_ids, topk_w, local_rank, chunk_counts, counts,
                                      route_counter, status, st);
  if (err != cudaSuccess) return err;
  // columns per work item: 1024, or down to 256 when there are few tokens,
  // so that the items fill the resident warps (8 CTAs of 8 warps per SM)
  int piece_cols = kGatherCols;
  while (piece_cols > 256 && static_cast<int64_t>(s.T) * ((s.H + piece_cols - 1) / piece_cols) <
                                 static_cast<int64_t>(num_sms) * 64)
    piece_cols /= 2;
  const int64_t items = static_cast<int64_t>(s.T) * ((s.H + piece_cols - 1) / piece_cols);
  const int64_t tail = static_cast<int64_t>(s.E) * kRowBlock / 256;  // enough threads for the padding rows
  int64_t blocks = (items + 7) / 8;  // 8 warps (items) per CTA
  if (blocks < tail) blocks = tail;
  if (blocks > 4096) blocks = 4096;
  // gathered bytes from which the gate/up GEMM launches after this kernel's
  // wait (measured: decode, 4 MB, 2 us faster; layers of 64 KB to 0.6 MB
  // 0.4 to 1.2 us slower)
  constexpr int64_t kLateTriggerBytes = int64_t(1) << 20;
  err = launch_pdl(permute_gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, s.T, s.H, s.E,
                   s.k, nch, static_cast<int64_t>(max_blocks_of(s)), static_cast<const int32_t*>(topk_ids),
                   static_cast<const int32_t*>(local_rank), counts,
                   static_cast<const int32_t*>(chunk_counts), X, Xp, scatter_idx, gather_idx, off_pad,
                   block_expert, num_blocks, route_counter, fwd_counters, n_fwd, piece_cols,
                   static_cast<int64_t>(s.T) * s.k * s.H * 2 >= kLateTriggerBytes ? 1 : 0, status);
  if (err != cudaSuccess) return err;
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

constexpr int64_t kNoAllocHistInts = int64_t(1) << 18;  // 1 MiB of int32 chunk histograms
constexpr int64_t kNoAllocHeadInts = 64;                  // 256 bytes ahead of them: the counter words
constexpr int64_t kNoAllocScratchInts = kNoAllocHeadInts + kNoAllocHistInts;

// [0]: the routing's chunk counter (zero when the module is loaded; every
// call leaves it at zero), [1]: the mark its scan leaves (cleared at the start
// of every call); [64 ..): the per-chunk expert histograms.
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
  if (static_cast<int64_t>(shape->E) * num_chunks_of(*shape) > kNoAllocHistInts) return MOE_ERR_SCRATCH_LIMIT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceRestore restore;
  st = device_ready(s, nullptr, &restore);  // the stream's device is current until this call returns
  if (st != MOE_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  int32_t* scratch = route_scratch_on_device(dev);
  if (scratch == nullptr) return MOE_ERR_CUDA;
  // Every chunk-histogram entry the scan and scatter read is written by the
  // first kernel of this call, so stale histograms need no clearing; the
  // chunk counter starts at zero (module load) and each call's second kernel
  // puts it back to zero.
  const cudaError_t e = launch_route(*shape, logits, topk_ids, topk_w, counts, off_pad, block_expert, num_blocks,
                                     gather_idx, scatter_idx, scratch + kNoAllocHeadInts,
                                     reinterpret_cast<uint32_t*>(scratch), /*status=*/nullptr, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
