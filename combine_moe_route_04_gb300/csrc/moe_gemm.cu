// moe_gemm.cu -- persistent, warp-specialised grouped GEMMs of the expert
// layer on the sm_103a tensor cores (tcgen05 + TMEM + TMA), and the row
// gather that fills their input.
//
// What they compute ("通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §1: gate/up
// GEMM -> SiLU -> down GEMM; "通算融合算子（三）：ThunderKittens 多卡编程与可融合的
// GEMM 模板" §4: rows grouped by expert, each group multiplies the weights of
// its own expert, tasks visited expert by expert):
//   up:   for each window A_w of expert e's rows (in permuted order) and each
//         256-column weight slice j,
//         G = A_w Wg[e][:, j], U = A_w Wu[e][:, j]  (float32 in TMEM)
//         h[w, j] = bf16(silu(G) * U)
//   down: Y[w, j] = bf16(h_w Wd[e][:, j]) for 512-column slices j.
// The row gather (scatter_rows_kernel) writes X[t] to each of token t's k
// permuted rows, reading every row of X once.
//
// Design (the roles and barrier lifetimes of "TIRx 与高性能GEMM (下)" Step 7,
// and the two-CTA MMA of its Step 8, re-keyed to expert row windows):
//   * a cluster of two CTAs on two SMs computes one tile = one window of an
//     expert's rows x 256 weight columns (up: of W_gate and of W_up) or 512
//     (down), with M=256 tcgen05.mma (cta_group::2).  The weights are the M
//     operand: per MMA CTA r holds 128 weight columns (N-major boxes read as
//     an MN-major A operand); the window's tokens are the N operand (N = real
//     rows rounded up to 16, at most 256), CTA r supplying tokens
//     [r N/2, (r+1) N/2).  Each CTA's TMEM holds two accumulators of 128
//     weight columns (lanes) x N tokens (columns), filled by two MMAs per K
//     step that share the token rows;
//   * an expert's rows are cut into equal windows so the tiles sharing a
//     weight tile run in step and read it from L2 together; padding beyond
//     the real rows costs at most 15 rows per window;
//   * tiles: each GEMM's clusters draw them from a counter in the workspace
//     (see the tile scheduler below), in expert-major order;
//   * warp 0 of each CTA, TMA producer: per 32-deep K stage, its weight
//     columns (two 32x64 boxes per accumulator, 128-byte swizzle: the up
//     GEMM loads W_gate and W_up, the down GEMM two neighbouring blocks of
//     W_down) and its token rows (a 128x32 box, or 64 / 80 rows for a short
//     window; 64-byte swizzle) into a ring of 9 stages of 24 KB; all loads
//     complete on CTA 0's full barriers;
//   * warp 1 allocates 512 TMEM columns in both CTAs; in CTA 0 one elected
//     lane issues the MMAs (the up GEMM issues a W_gate and a W_up MMA per K
//     step into accumulators g | u, so SiLU(g)*u meets in one thread) and
//     commits stages back to both producers and results to both epilogues;
//   * warps 2-9 of each CTA drain the accumulator (thread = weight column;
//     two warps per 32-lane TMEM quarter, taking its 32-token chunks in
//     turn) into registers, release it on CTA 0's accumulator-empty barrier
//     once their last TMEM load has landed, and write their column down the
//     window's output rows (in the up GEMM neighbouring lanes swap token
//     halves and store two columns of one token each).  The two accumulators
//     fill TMEM (one set);
//   * inside one forward the two GEMMs hand over per window: the gate/up
//     epilogue counts each stored tile on its window's counter, and the down
//     GEMM's producers wait for their window's count instead of for the whole
//     gate/up grid (see the kernel's entry).  Where the gate/up GEMM is one
//     wave of tiles, a down producer loads the weight slices of its tile's
//     first stages while it waits and the token rows after.
// Every wait on an mbarrier or a counter is bounded; on a timeout the kernel
// records it in the status word, the roles stop, in-flight copies and MMAs
// are drained (bounded) and TMEM is freed before exit.
#include <cstdint>
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BK = 32;                           // K per pipeline stage
constexpr int B_BOX_BYTES = BK * 64 * 2;         // 4 KB: 32 k-rows x 64 columns (128-byte swizzle)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;

constexpr int MAX_E = 256;

// Epilogue warps: two per 32-lane TMEM quarter (a warp may read only the
// quarter warp_id % 4), draining and storing alternate 32-token chunks.
constexpr int S_EPI_WARPS = 8;
constexpr int S_EPI_SPLIT = S_EPI_WARPS / 4;             // warps sharing a lane quarter

// OR-vote over the epilogue threads (named barrier 2).
__device__ __forceinline__ bool vote_any_epi(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 2, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(flag ? 1u : 0u), "n"(S_EPI_WARPS * 32)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// Token-window ("swap") orientation.  The weights are the M=256 MMA
// operand (CTA r holds 128 weight columns, N-major boxes read as an MN-major
// A operand) and the expert's tokens are the N operand: a tile is one window
// of up to 256 consecutive rows of one expert times 256 weight columns, and
// N = the window's real row count rounded up to 16, so an expert wastes fewer
// than 16 rows per window instead of the rest of a 128-row block.  In
// cta_group::2 the N operand is split between the CTAs: CTA r supplies tokens
// [r N/2, (r+1) N/2) of the window, and both CTAs' TMEM hold all N token
// columns for their own 128 weight columns (TMEM lane = weight column).
//   up:   two MMAs per K step, W_gate columns into accumulator g and the same
//         W_up columns into accumulator u, so a thread owns g and u of one
//         column for every token; h = SiLU(g) * u.
//   down: two MMAs per K step into two accumulators of neighbouring
//         128-column blocks of W_down (a 512-column tile per pair).
// 512 TMEM columns = the two accumulators: one set, so the epilogue drain is
// not overlapped with the next tile's MMAs (measured: double-buffering the
// down GEMM's single 256-column accumulator instead was slower, its stages
// then needing more shared-memory bandwidth than the data path has).
// The epilogue holds one weight column for its share of the window's tokens
// and writes it down the output rows (the transpose happens on the way out).
constexpr int S_TOK = 256;                               // max tokens per window
static_assert(S_TOK == kWindowRows, "window size shared with the workspace layout");
constexpr int S_TOK_BOX = 128;                           // token rows per TMA box (per CTA)
constexpr int S_W_BYTES = 2 * B_BOX_BYTES;               // 8 KB: 32 k-rows x 128 weight columns
constexpr int S_T_BYTES = S_TOK_BOX * BK * 2;            // 8 KB: 128 token rows x 32 k (64-byte swizzle)
constexpr int S_THREADS = (2 + S_EPI_WARPS) * 32;        // producer, MMA, epilogue warps
constexpr int S_GROUP_WINDOWS = 4;                       // L2 grouping of windows inside an expert
constexpr int S_TILE_RING = 8;                           // tile indices in flight from the scheduler
// readers of each tile index: CTA 0's MMA lane and its epilogue warps, CTA
// 1's producer lane and its epilogue warps (CTA 0's producer lane is the
// scheduler)
constexpr int S_TILE_READERS = 1 + S_EPI_WARPS + 1 + S_EPI_WARPS;

// Both GEMMs run two 128-column accumulators per CTA that share each K
// step's token rows: the up GEMM's gate and up columns, the down GEMM's two
// neighbouring 128-column blocks (so a down tile is 512 weight columns, 256
// per CTA).  A stage is 24 KB of loads for two MMAs per 16-deep K substep:
// the token rows, read by both tensor cores of the pair, serve two
// accumulators, which is the least shared-memory traffic (TMA writes + MMA
// operand reads) per FLOP that the MMA shape and TMEM allow.  The two
// accumulators fill TMEM, so there is one accumulator set and the epilogue
// drain is not overlapped.
template <bool kUp>
struct SwapCfg {
  static constexpr int TILE_COLS = kUp ? 256 : 512;      // output columns per tile
  static constexpr int STAGE_BYTES = 2 * S_W_BYTES + S_T_BYTES;  // 24 KB
  static constexpr int STAGES = 9;
  static constexpr int NBUF = 1;                         // accumulator sets in TMEM
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NBUF + 1 + 2 * S_TILE_RING;
  static constexpr int WIN_OFF = BAR_OFF + NUM_BARS * 8 + 16;
  static constexpr int TILE_OFF = (WIN_OFF + (MAX_E + 1) * 4 + 15) / 16 * 16;
  static constexpr int CNT_OFF = TILE_OFF + S_TILE_RING * 4;     // counts[e], copied at entry
  static constexpr int OFFP_OFF = CNT_OFF + MAX_E * 4;           // off_pad[e], copied at entry
  static constexpr int BYTES = OFFP_OFF + (MAX_E + 1) * 4;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(ALLOC <= 232448, "shared memory budget (window kernel)");
};

struct WinCoord {
  int e;      // expert
  int j;      // 256-column weight tile
  int row0;   // first permuted row of the window
  int rows;   // real rows in the window (1..256)
  int wid;    // window index over all experts (w_off[e] + window)
  bool ok;
};

// An expert's c rows are cut into nw = ceil(c / 256) windows of equal size S
// = round16(ceil(c / nw)) (the last may be shorter), so the windows that
// share a weight tile take the same time and read it from L2 together.
// Tile t: expert e (windows w_off[e] .. w_off[e+1]), then groups of
// S_GROUP_WINDOWS windows, then weight tile, then the window in the group.
__device__ __forceinline__ WinCoord decode_window(int tile, int NT, int E, const int32_t* s_win_off,
                                                  const int32_t* s_offp, const int32_t* s_cnt, int64_t max_rows) {
  WinCoord c{0, 0, 0, 0, 0, false};
  const int q = tile / NT;
  int lo = 0, hi = E;  // last e with s_win_off[e] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_win_off[mid] <= q) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  if (e >= E) return c;
  const int nw = s_win_off[e + 1] - s_win_off[e];
  const int local = tile - NT * s_win_off[e];
  if (nw <= 0 || local < 0 || local >= NT * nw) return c;
  const int g = local / (NT * S_GROUP_WINDOWS);
  const int rem = local - g * NT * S_GROUP_WINDOWS;
  const int gs = min(S_GROUP_WINDOWS, nw - g * S_GROUP_WINDOWS);
  const int w = g * S_GROUP_WINDOWS + rem % gs;
  const int cnt = s_cnt[e];
  const int S = ((cnt + nw - 1) / nw + 15) / 16 * 16;
  c.e = e;
  c.j = rem / gs;
  c.row0 = s_offp[e] + S * w;
  c.rows = min(S, cnt - S * w);
  c.wid = s_win_off[e] + w;
  // the window's rows lie inside the expert's padded range
  const int pad_end = s_offp[e + 1];
  c.ok = c.rows > 0 && c.rows <= S_TOK && c.row0 >= 0 && c.row0 + c.rows <= pad_end && pad_end <= max_rows &&
         c.j < NT;
  return c;
}

// Dynamic tile scheduler.  Cluster c starts on tile c; after that CTA 0's
// producer lane draws tile indices from a counter in global memory (tile
// nclusters + the counter's old value, atomicAdd, in tile order, so the
// windows that share a weight tile are still drawn together) and publishes
// each into a
// ring in both CTAs' shared memory; every other role of the pair reads the
// same sequence from its own CTA's ring.  A cluster draws and publishes its
// next tile when it starts the current one, so the index is in place a whole
// tile before any role needs it, and clusters that got smaller windows take
// more tiles.  The cluster that finishes drawing last resets the counter for
// the next launch.
struct TileRing {
  uint64_t* full;        // [S_TILE_RING], this CTA: one arrival (the scheduler)
  uint64_t* empty;       // [S_TILE_RING], used in CTA 0: S_TILE_READERS arrivals
  volatile int32_t* idx; // [S_TILE_RING], this CTA
};

// Reader side: the index of the n-th tile of this cluster; -1 when a bounded
// wait gave up.  CTA 0's readers synchronise at CTA scope, CTA 1's at cluster
// scope.  With release == false the caller releases the slot (ring_release).
__device__ __forceinline__ void ring_release(const TileRing& r, uint32_t n, uint32_t rank, uint32_t empty0_cluster) {
  const uint32_t slot = n % S_TILE_RING;
  if (rank == 0) mbar_arrive(&r.empty[slot]);
  else mbar_arrive_cluster(empty0_cluster + 8u * slot);
}
__device__ __forceinline__ int ring_take(const TileRing& r, uint32_t n, uint32_t rank, uint32_t empty0_cluster,
                                         bool release, volatile int* abort, uint32_t* status) {
  const uint32_t slot = n % S_TILE_RING;
  const uint32_t ph = (n / S_TILE_RING) & 1u;
  const bool ok = rank == 0 ? mbar_wait<false>(&r.full[slot], ph, abort, status)
                            : mbar_wait<true>(&r.full[slot], ph, abort, status);
  if (!ok) return -1;
  const int t = r.idx[slot];
  if (release) ring_release(r, n, rank, empty0_cluster);
  return t;
}

// Scheduler side (CTA 0): publish the n-th tile index to both CTAs.
__device__ __forceinline__ bool ring_put(const TileRing& r, uint32_t n, int tile, volatile int* abort,
                                         uint32_t* status) {
  const uint32_t slot = n % S_TILE_RING;
  if (!mbar_wait(&r.empty[slot], ((n / S_TILE_RING) & 1u) ^ 1u, abort, status)) return false;
  r.idx[slot] = tile;
  mbar_arrive(&r.full[slot]);
  const uint32_t remote_idx = map_to_cta(const_cast<int32_t*>(&r.idx[slot]), 1);
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote_idx), "r"(tile) : "memory");
  mbar_arrive_cluster(map_to_cta(&r.full[slot], 1));
  return true;
}

template <bool kUp>
__global__ void __launch_bounds__(S_THREADS, 1)
    grouped_gemm_window_kernel(const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmT64,
                               const __grid_constant__ CUtensorMap tmT80, const __grid_constant__ CUtensorMap tmW0,
                               const __grid_constant__ CUtensorMap tmW1, uint16_t* __restrict__ D,
                               const int32_t* __restrict__ off_pad, const int32_t* __restrict__ counts, int E,
                               int K, int NT, int N_out, int64_t max_rows, uint32_t* __restrict__ status,
                               uint32_t* __restrict__ sched, uint32_t* __restrict__ win_done, uint32_t win_target) {
  using C = SwapCfg<kUp>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sStage = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = bars + 2 * C::STAGES + C::NBUF;
  uint64_t* drain = bars + 2 * C::STAGES + 2 * C::NBUF;
  const TileRing ring{bars + 2 * C::STAGES + 2 * C::NBUF + 1, bars + 2 * C::STAGES + 2 * C::NBUF + 1 + S_TILE_RING,
                      reinterpret_cast<volatile int32_t*>(smem + C::TILE_OFF)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_win_off = reinterpret_cast<int32_t*>(smem + C::WIN_OFF);
  int32_t* s_cnt = reinterpret_cast<int32_t*>(smem + C::CNT_OFF);
  int32_t* s_offp = reinterpret_cast<int32_t*>(smem + C::OFFP_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  // Per-window hand-off inside one forward (win_done set): the gate/up GEMM
  // counts each window's finished tiles, and the down GEMM that follows it
  // waits for its windows' counts instead of for the whole grid, so its
  // clusters start on the SMs this grid frees.  This grid then lets it launch
  // only after its own wait below (the rows and routing it reads are final;
  // the routing cleared the counts); the down GEMM lets the combine launch
  // after its producers' last loads.
  const bool tracked = win_done != nullptr;
  if (!tracked) pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::NBUF; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * S_EPI_WARPS);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    for (int i = 0; i < S_TILE_RING; ++i) {
      mbar_init(&ring.full[i], 1);
      mbar_init(&ring.empty[i], S_TILE_READERS);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tmap(&tmT);
    prefetch_tmap(&tmT64);
    prefetch_tmap(&tmT80);
    prefetch_tmap(&tmW0);
    prefetch_tmap(&tmW1);
  }
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA arrival
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }

  if (kUp || !tracked) pdl_wait();
  if (kUp && tracked) pdl_launch_dependents();
  if (warp == 2) {
    // windows per expert (ceil(count / 256)) -> exclusive scan, E <= 256
    constexpr int per = MAX_E / 32;
    int loc[per];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      int nw = 0;
      if (e < E) {
        const int cnt = __ldg(counts + e);
        s_cnt[e] = cnt;  // the tile decoder's copy
        nw = cnt > 0 ? (cnt + S_TOK - 1) / S_TOK : 0;
      }
      loc[i] = nw;
      sum += nw;
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
      if (e <= E) s_win_off[e] = run;
      run += loc[i];
    }
    if (lane == 31 && 32 * per == E) s_win_off[E] = incl;
  } else if (warp == 3) {
    // the tile decoder's copy of the padded offsets
    for (int e = lane; e <= E; e += 32) s_offp[e] = __ldg(off_pad + e);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = NT * s_win_off[E];
  const int KB = K / BK;
  const int nclusters = gridDim.x >> 1;
  const uint32_t full0 = map_to_cta(full, 0);
  const uint32_t tempty0 = map_to_cta(tempty, 0);
  const uint32_t rempty0 = map_to_cta(ring.empty, 0);

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer (both CTAs)
    if (elect_one_sync()) {
      const uint64_t pol_t = policy_evict_last();
      // the status word when this forward began (recorded by its routing)
      const uint32_t status_before = (!kUp && tracked) ? __ldcg(status + kStatusSnapshotIndex) : 0u;
      const uint64_t pol_wn = policy_evict_normal();
      const uint64_t pol_wf = policy_evict_first();
      uint32_t it = 0;
      bool stop = false;
      // down GEMM in a forward whose gate/up GEMM is one wave of tiles (at
      // most one per CTA pair the GPU holds; win_target counts one arrival
      // per epilogue warp of both CTAs for each of a window's column tiles):
      // its CTAs wait for windows on SMs the gate/up GEMM leaves idle, so
      // each tile's first weight slices are loaded during that wait.
      const int64_t up_tiles = static_cast<int64_t>(s_win_off[E]) * (win_target / (2u * S_EPI_WARPS));
      const bool early_weights = !kUp && tracked && up_tiles <= static_cast<int64_t>(num_sm_ids() / 2);
      // first ring use retired by the abort path below (left out of the drain)
      uint32_t retired_from = 0xFFFFFFFFu;
      // each cluster's first tile is its cluster index (no draw in front of
      // its first loads); CTA 0 draws the pair's later tiles and publishes
      // them; CTA 1 reads them
      int tile;
      if (rank == 0) {
        tile = static_cast<int>(blockIdx.x >> 1);
        stop = !ring_put(ring, 0, tile, abort_flag, status);
      } else {
        tile = ring_take(ring, 0, rank, rempty0, true, abort_flag, status);
      }
      for (uint32_t n = 0; !stop && tile >= 0 && tile < total_tiles; ++n) {
        // CTA 0 draws the next tile now without waiting for the value, and
        // publishes it halfway through this tile's loads.  Draws follow the
        // nclusters first tiles, one per tile processed, so a cleared counter
        // yields nclusters .. total_tiles + nclusters - 1; a larger value
        // means the counter was not cleared and ends the sequence.
        const uint32_t raw_next = rank == 0 ? atomicAdd(sched, 1u) : 0u;
        int next = total_tiles;
        bool published = rank != 0;
        auto publish = [&]() {
          const uint64_t t = static_cast<uint64_t>(nclusters) + raw_next;
          next = t < static_cast<uint64_t>(total_tiles + nclusters) ? static_cast<int>(t) : total_tiles;
          if (static_cast<uint64_t>(next) != t) record_status(status, kStatusBounds);
          published = true;
          return ring_put(ring, n + 1, next, abort_flag, status);
        };
        const WinCoord c = decode_window(tile, NT, E, s_win_off, s_offp, s_cnt, max_rows);
        if (!c.ok) record_status(status, kStatusBounds);
        // a one-window expert reads this weight tile once: evict it first and
        // keep the rows, h and Y in L2; windows sharing a tile read it together
        const uint64_t pol_w = (s_win_off[c.e + 1] - s_win_off[c.e]) == 1 ? pol_wf : pol_wn;
        const int n_half = ((c.rows + 15) / 16) * 8;                   // tokens this CTA supplies
        const int trow = c.row0 + static_cast<int>(rank) * n_half;     // its first token row
        const int n0 = c.j * C::TILE_COLS + (C::TILE_COLS / 2) * static_cast<int>(rank);  // first weight column
        // the token box: 128 rows, or 64 / 80 when this CTA supplies no more
        // (short windows: fewer shared-memory bytes per stage; the MMA reads
        // only the first n_half rows either way)
        const CUtensorMap* tmap = &tmT;
        int box_rows = S_TOK_BOX;
        if (n_half <= 64) {
          tmap = &tmT64;
          box_rows = 64;
        } else if (n_half <= 80) {
          tmap = &tmT80;
          box_rows = 80;
        }
        const uint32_t stage_tx = 2u * static_cast<uint32_t>(2 * S_W_BYTES + box_rows * BK * 2);
        // stage kb of this tile: the weight tile's K slice, then the token rows
        auto load_weights = [&](uint32_t s, int kb) {
          uint8_t* st = sStage + s * C::STAGE_BYTES;
          const uint32_t fb = full0 + 8u * s;
          const int k0 = c.e * K + kb * BK;
          tma_load_2d_pair(st, &tmW0, fb, n0, k0, pol_w);
          tma_load_2d_pair(st + B_BOX_BYTES, &tmW0, fb, n0 + 64, k0, pol_w);
          if (kUp) {  // the same columns of W_up
            tma_load_2d_pair(st + S_W_BYTES, &tmW1, fb, n0, k0, pol_w);
            tma_load_2d_pair(st + S_W_BYTES + B_BOX_BYTES, &tmW1, fb, n0 + 64, k0, pol_w);
          } else {  // the CTA's next 128 columns of W_down
            tma_load_2d_pair(st + S_W_BYTES, &tmW0, fb, n0 + 128, k0, pol_w);
            tma_load_2d_pair(st + S_W_BYTES + B_BOX_BYTES, &tmW0, fb, n0 + 192, k0, pol_w);
          }
        };
        auto load_tokens = [&](uint32_t s, int kb) {
          tma_load_2d_pair(sStage + s * C::STAGE_BYTES + 2 * S_W_BYTES, tmap, full0 + 8u * s, kb * BK, trow, pol_t);
        };
        // claims the next ring stage for this tile (its empty wait, then the
        // expected bytes of both CTAs' loads on CTA 0's full barrier)
        auto claim = [&](uint32_t s) {
          if (!mbar_wait(&empty[s], ((it / C::STAGES) & 1u) ^ 1u, abort_flag, status)) return false;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], stage_tx);
          return true;
        };
        // down GEMM in a forward: this window's h rows are complete once all
        // its gate/up tiles have counted in.  The weights do not depend on
        // them: with early_weights the first stages' weight slices (as many
        // as the ring holds) are loaded before the wait and their token rows
        // after it.
        const int pre = (early_weights && c.ok) ? (KB < static_cast<int>(C::STAGES) ? KB : static_cast<int>(C::STAGES)) : 0;
        const uint32_t it0 = it;
        // If this CTA stops with stages claimed before the wait (weights in
        // flight, token rows not loaded), it loads their token rows anyway
        // (in range; the values are not used), which completes the stages'
        // full barriers, and CTA 0 waits for those: no copy is pending when
        // the pair exits (CTA 1 is held by the final cluster barrier until
        // CTA 0 gets there).  The MMA issuer may or may not consume these
        // stages, so the drain leaves them out; their earlier uses were
        // consumed before they were claimed.
        auto retire_claimed = [&]() {
          const uint32_t n = it - it0;
          for (uint32_t u = 0; u < n; ++u) load_tokens((it0 + u) % C::STAGES, static_cast<int>(u));
          if (rank == 0) {
            for (uint32_t u = it0; u < it; ++u) {
              int no_abort = 0;
              mbar_wait(&full[u % C::STAGES], (u / C::STAGES) & 1u, &no_abort, status);
            }
          }
          if (n > 0) retired_from = it0;
        };
        for (int kb = 0; kb < pre; ++kb, ++it) {
          if (!published && kb == KB / 2 && !publish()) {
            stop = true;
            break;
          }
          if (!claim(it % C::STAGES)) {
            stop = true;
            break;
          }
          load_weights(it % C::STAGES, kb);
        }
        if (stop) {
          retire_claimed();
          break;
        }
        if (!kUp && tracked && c.ok &&
            !wait_counter_at_least(win_done + c.wid, win_target, abort_flag, status, status_before)) {
          retire_claimed();
          stop = true;
          break;
        }
        for (int kb = 0; kb < pre; ++kb) load_tokens((it0 + kb) % C::STAGES, kb);
        for (int kb = pre; c.ok && kb < KB; ++kb, ++it) {
          if (!published && kb == KB / 2 && !publish()) {
            stop = true;
            break;
          }
          const uint32_t s = it % C::STAGES;
          if (!claim(s)) {
            stop = true;
            break;
          }
          load_weights(s, kb);
          load_tokens(s, kb);
        }
        if (stop) break;
        if (!published && !publish()) break;
        tile = rank == 0 ? next : ring_take(ring, n + 1, rank, rempty0, true, abort_flag, status);
      }
      if (rank == 0) {
        // this cluster has drawn its last index; the last cluster to get here
        // clears the counter for the next launch
        __threadfence();
        if (atomicAdd(sched + 1, 1u) == static_cast<uint32_t>(nclusters - 1)) {
          atomicExch(sched, 0u);
          atomicExch(sched + 1, 0u);
        }
      }
      // down GEMM of a forward: the combine may launch once every producer
      // has issued its last loads (launched at entry, its CTAs would wait on
      // SMs through the whole GEMM; at exit, its launch would not overlap)
      if (!kUp && tracked) pdl_launch_dependents();
      const uint32_t nst = it < C::STAGES ? it : C::STAGES;
      for (uint32_t s = 0; s < nst; ++s) {
        const uint32_t last = s + C::STAGES * ((it - 1 - s) / C::STAGES);
        if (last >= retired_from) continue;  // retired above: copies landed, earlier uses consumed
        int no_abort = 0;
        mbar_wait(&empty[s], (last / C::STAGES) & 1u, &no_abort, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer (CTA 0)
    if (rank == 0 && elect_one_sync()) {
      // M=256 (weights, MN-major A), N from the window, A MN-major, B K-major
      constexpr uint32_t idesc_base = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((256u >> 4) << 24);
      uint32_t it = 0;
      uint32_t tcount = 0;
      bool stop = false;
      for (uint32_t n = 0; !stop; ++n) {
        const int tile = ring_take(ring, n, rank, rempty0, true, abort_flag, status);
        if (tile < 0 || tile >= total_tiles) break;
        const WinCoord c = decode_window(tile, NT, E, s_win_off, s_offp, s_cnt, max_rows);
        if (!c.ok) continue;
        const uint32_t N = static_cast<uint32_t>(((c.rows + 15) / 16) * 16);
        const uint32_t idesc = idesc_base | ((N >> 3) << 17);
        const uint32_t a = 0;               // one accumulator set (g | u, or the two blocks)
        const uint32_t aph = tcount & 1u;
        if (!mbar_wait(&tempty[a], aph ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + a * ACC_COLS;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, status)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(sStage + s * C::STAGE_BYTES);
          const uint32_t tk = st + 2 * S_W_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A (weights, this CTA's 128 columns): MN-major, 128-byte swizzle,
            // 64-column boxes 4 KB apart, 8-row K groups 1 KB apart, K step 2 KB.
            // B (tokens, this CTA's N/2 rows): K-major, 64-byte swizzle, 8-row
            // groups 512 B apart, K step 32 B.
            const uint64_t bdesc = smem_desc(tk + kk * 32, 16, 512, kSwizzle64B);
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            tc_mma_f16_pair(d, smem_desc(st + kk * 2048, B_BOX_BYTES, 1024, kSwizzle128B), bdesc, idesc, acc);
            tc_mma_f16_pair(d + 256, smem_desc(st + S_W_BYTES + kk * 2048, B_BOX_BYTES, 1024, kSwizzle128B),
                              bdesc, idesc, acc);
          }
          tc_commit_pair(&empty[s], 0x3);
        }
        if (stop) break;
        tc_commit_pair(&tfull[a], 0x3);
        ++tcount;
      }
      tc_commit_pair(drain, 0x1);
      int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue (both CTAs)
    // thread = TMEM lane = weight column `col` of this CTA's 128: it holds
    // that column for its warp's share of the window's tokens and writes it
    // down those output rows
    const int q = warp & 3;                                   // TMEM lane quarter
    const int col = q * 32 + lane;
    constexpr int CH_PER = S_TOK / 32 / S_EPI_SPLIT;          // 32-token chunks per warp (at most)
    // the quarter's warps take its 32-token chunks in turn (chunk half,
    // half + S_EPI_SPLIT, ...), so a short window still splits evenly
    const int half = (warp - 2) / 4;
    uint32_t tcount = 0;
    for (uint32_t n = 0;; ++n) {
      const int tile = ring_take(ring, n, rank, rempty0, false, abort_flag, status);
      __syncwarp();
      if (lane == 0) ring_release(ring, n, rank, rempty0);
      if (vote_any_epi(tile < 0)) break;
      if (tile >= total_tiles) break;
      const WinCoord c = decode_window(tile, NT, E, s_win_off, s_offp, s_cnt, max_rows);
      if (!c.ok) continue;
      const uint32_t a = 0;
      const uint32_t aph = tcount & 1u;
      const bool ok = mbar_wait(&tfull[a], aph, abort_flag, status);
      if (vote_any_epi(!ok)) break;
      tc_fence_after();
      const int nchunks = (c.rows + 31) / 32;       // 32-token TMEM column chunks holding real rows
      const int mine = nchunks > half ? (nchunks - half + S_EPI_SPLIT - 1) / S_EPI_SPLIT : 0;
      // the accumulator is free once this warp's last TMEM load has landed:
      // every warp arrives then, before converting that chunk
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0 + 8u * a);
      };
      if (mine == 0) release();
      uint32_t packed[CH_PER * 16];                 // bf16 pairs (token 2i, 2i+1 of chunk cl) of this column
      uint32_t packed1[kUp ? 1 : CH_PER * 16];      // down: the second accumulator's column
      const uint32_t tbase = tmem_base + a * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
      for (int cl = 0; cl < CH_PER; ++cl) {
        const int ch = half + S_EPI_SPLIT * cl;
        if (cl < mine) {
          if constexpr (kUp) {
            uint32_t gv[32], uv[32];
            tmem_ld_32x32b_x32(tbase + ch * 32, gv);
            tmem_ld_32x32b_x32(tbase + 256 + ch * 32, uv);
            tmem_ld_wait();
            if (cl == mine - 1) release();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(gv[2 * i]), g1 = __uint_as_float(gv[2 * i + 1]);
              const float u0 = __uint_as_float(uv[2 * i]), u1 = __uint_as_float(uv[2 * i + 1]);
              // silu(g) = g * sigmoid(g) on the SFU (a few float32 ulps, far
              // below the bf16 rounding of h; g < -88 gives the limit 0)
              const float h0 = g0 * __fdividef(1.0f, 1.0f + __expf(-g0)) * u0;
              const float h1 = g1 * __fdividef(1.0f, 1.0f + __expf(-g1)) * u1;
              packed[cl * 16 + i] = pack_bf16x2(h0, h1);
            }
          } else {  // down: one accumulator at a time (register pressure)
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + ch * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[cl * 16 + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            tmem_ld_32x32b_x32(tbase + 256 + ch * 32, v);
            tmem_ld_wait();
            if (cl == mine - 1) release();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed1[cl * 16 + i] =
                  pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          }
        }
      }
      ++tcount;
      // out[row0 + t][tile columns + col] for the window's real rows.
      // Up GEMM: neighbouring lanes (columns 2m, 2m+1) swap halves of their
      // token pairs, so the even lane stores token 2i and the odd lane token
      // 2i+1, each as two adjacent columns (4 bytes): half as many stores.
      // Down GEMM: one column per lane per accumulator, 2-byte stores.
      const int colg = c.j * C::TILE_COLS + (C::TILE_COLS / 2) * static_cast<int>(rank) + col;
      if constexpr (!kUp) {
        // one accumulator's column down the rows; a column past N_out (a
        // last tile partly outside) is skipped, uniformly across the warp
        auto store_column = [&](const uint32_t (&pk)[CH_PER * 16], int cg) {
          if (cg >= N_out) return;
          // chunk cl starts S_EPI_SPLIT * 32 * cl tokens after the warp's first
          uint16_t* dst = D + static_cast<int64_t>(c.row0 + half * 32) * N_out + cg;
          const int rem = c.rows - half * 32;
#pragma unroll
          for (int cl = 0; cl < CH_PER; ++cl) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int t = S_EPI_SPLIT * 32 * cl + 2 * i;
              if (t < rem) {
                const uint32_t v = pk[cl * 16 + i];
                dst[static_cast<int64_t>(t) * N_out] = static_cast<uint16_t>(v & 0xFFFFu);
                if (t + 1 < rem) dst[static_cast<int64_t>(t + 1) * N_out] = static_cast<uint16_t>(v >> 16);
              }
            }
          }
        };
        store_column(packed, colg);
        store_column(packed1, colg + 128);  // the second accumulator: 128 columns further
      } else if (colg < N_out) {            // uniform across the warp (N_out % 128 == 0)
        const int odd = lane & 1;
        uint32_t* dst =
            reinterpret_cast<uint32_t*>(D + static_cast<int64_t>(c.row0 + half * 32 + odd) * N_out + (colg & ~1));
        const int rem = c.rows - half * 32;
#pragma unroll
        for (int cl = 0; cl < CH_PER; ++cl) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int t = S_EPI_SPLIT * 32 * cl + 2 * i;
            if (t < rem) {  // uniform across the warp
              const uint32_t v_mine = packed[cl * 16 + i];
              const uint32_t other = __shfl_xor_sync(0xffffffffu, v_mine, 1);
              const uint32_t v = odd ? __byte_perm(other, v_mine, 0x7632) : __byte_perm(v_mine, other, 0x5410);
              if (t + odd < rem) dst[static_cast<int64_t>(t / 2) * N_out] = v;  // two rows = N_out words
            }
          }
        }
      }
      if (kUp && tracked) {
        // this warp's part of the window is written: count it (the warp's
        // stores are ordered before the fence by the warp barrier)
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_gpu();  // release: the warp's stores before the count
          atomicAdd(win_done + c.wid, 1u);
        }
      }
    }
  }

  // The down GEMM of a forward skipped griddepcontrol.wait at entry; it waits
  // here, once its work is done, so that its completion implies that of the
  // whole gate/up grid (including the last cluster's reset of the gate/up
  // tile counter): every later kernel of the stream that waits on this grid
  // then finds the gate/up GEMM finished too.  By now the gate/up grid has
  // stored every window, so this wait is short.
  if (!kUp && tracked) pdl_wait();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Fills Xp (the token rows in permuted order) token by token: a warp takes
// one token and a 1024-column chunk, reads that piece of X once and writes it
// to the token's k rows (scatter_idx).  Each row of X is read from memory
// once, in order, however many experts picked it; padding rows of Xp are left
// untouched (the GEMM never stores their results).
__global__ void scatter_rows_kernel(const uint16_t* __restrict__ X, const int32_t* __restrict__ scatter_idx,
                                    int64_t max_rows, int T, int H, int k, uint16_t* __restrict__ Xp,
                                    uint32_t* __restrict__ status) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  constexpr int CH = kGatherCols;  // columns per work item: 16 bytes x 4 per lane
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = tid >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int nchunk = (H + CH - 1) / CH;
  const int64_t items = static_cast<int64_t>(T) * nchunk;
  for (int64_t item = warp0; item < items; item += nwarps) {
    const int t = static_cast<int>(item / nchunk);
    const int c0 = static_cast<int>(item % nchunk) * CH;
    int my_row = -1;  // lane j < k: row of (t, j)
    if (lane < k) {
      const int32_t r = __ldg(scatter_idx + static_cast<int64_t>(t) * k + lane);
      if (r >= 0 && r < max_rows) my_row = r;
      else record_status(status, kStatusBounds);
    }
    const int nv = min(CH, H - c0) / 8;  // 16-byte vectors in this chunk (H % 128 == 0)
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

template <bool kUp>
cudaError_t launch_gemm(const moe_shape& s, const GemmMaps& maps, uint16_t* D, const int32_t* off_pad,
                        const int32_t* counts, uint32_t* status, uint32_t* sched, uint32_t* win_done,
                        int num_sms, cudaStream_t st) {
  using C = SwapCfg<kUp>;
  // the shared-memory opt-in, once per device (host threads may race here)
  static bool attr_done[64] = {};
  static std::mutex attr_mu;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (dev >= 64 || !attr_done[dev]) {
      err = cudaFuncSetAttribute(grouped_gemm_window_kernel<kUp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::ALLOC);
      if (err != cudaSuccess) return err;
      if (dev < 64) attr_done[dev] = true;
    }
  }
  // 256 (up) / 512 (down) weight columns per tile; a last tile that reaches
  // past I or H is partly outside: TMA zero-fills those weight columns and
  // their stores are skipped
  const int NT = kUp ? (s.I + 255) / 256 : (s.H + C::TILE_COLS - 1) / C::TILE_COLS;
  const int K = kUp ? s.H : s.I;
  const int64_t max_tiles = max_windows_of(s) * NT;
  // a window's h rows are complete when every epilogue warp of both CTAs has
  // counted each of its gate/up tiles
  const uint32_t win_target = 2u * S_EPI_WARPS * static_cast<uint32_t>((s.I + 255) / 256);
  int64_t clusters = num_sms / 2;
  if (max_tiles < clusters) clusters = max_tiles;
  if (clusters <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  cfg.blockDim = dim3(S_THREADS);
  cfg.dynamicSmemBytes = C::ALLOC;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_window_kernel<kUp>, maps.a, maps.a64, maps.a80, maps.b0, maps.b1, D,
                            off_pad, counts, s.E, K, NT, kUp ? s.I : s.H, max_rows_of(s), status, sched, win_done,
                            win_target);
}

}  // namespace

cudaError_t launch_scatter_rows(const moe_shape& s, const uint16_t* X, const int32_t* scatter_idx, uint16_t* Xp,
                                uint32_t* status, cudaStream_t st) {
  const int64_t items = static_cast<int64_t>(s.T) * gather_pieces_of(s);
  int64_t blocks = (items + 7) / 8;  // 8 warps (items) per CTA
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(scatter_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, X, scatter_idx,
                    max_rows_of(s), s.T, s.H, s.k, Xp, status);
}

cudaError_t launch_gemm_up(const moe_shape& s, const GemmMaps& maps, uint16_t* h, const int32_t* off_pad,
                           const int32_t* counts, uint32_t* status, uint32_t* sched, uint32_t* win_done,
                           int num_sms, cudaStream_t st) {
  return launch_gemm<true>(s, maps, h, off_pad, counts, status, sched, win_done, num_sms, st);
}

cudaError_t launch_gemm_down(const moe_shape& s, const GemmMaps& maps, uint16_t* Y, const int32_t* off_pad,
                             const int32_t* counts, uint32_t* status, uint32_t* sched, uint32_t* win_done,
                             int num_sms, cudaStream_t st) {
  return launch_gemm<false>(s, maps, Y, off_pad, counts, status, sched, win_done, num_sms, st);
}

}  // namespace moe
