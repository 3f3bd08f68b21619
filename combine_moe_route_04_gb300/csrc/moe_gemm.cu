// moe_gemm.cu -- persistent, warp-specialised grouped GEMMs of the expert
// layer on the sm_103a tensor cores (tcgen05 + TMEM + TMA), and the row
// gather that feeds the gate/up GEMM.
//
// What they compute ("通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §1: gate/up
// GEMM -> SiLU -> down GEMM; "通算融合算子（三）：ThunderKittens 多卡编程与可融合的
// GEMM 模板" §4: each 128-row block multiplies the weights of its own expert,
// tasks visited expert by expert):
//   up:   for each 128-row block b of expert e and each 128-column slice j,
//         G = A_b Wg[e][:, j], U = A_b Wu[e][:, j]  (float32 in TMEM)
//         h[b, j] = bf16(silu(G) * U)
//   down: Y[b, j] = bf16(h_b Wd[e][:, j]) for 256-column slices j.
//
// Design (the roles and barrier lifetimes of "TIRx 与高性能GEMM (下)" Step 7,
// re-keyed to expert blocks; the B-tile sharing of its Step 9 done inside one
// CTA):
//   * a tile is a PAIR of 128-row blocks of the same expert (the second may be
//     absent) times one 256-column MMA tile: both blocks multiply the same B
//     tile, which cuts the bytes each SM must load per MMA clock by a third;
//   * warp 0, TMA producer: per 32-deep K stage, A of each block (128x32,
//     64-byte swizzle) and B (32x256 as four 32x64 boxes, N-major, 128-byte
//     swizzle) into a 6-stage SMEM ring guarded by full/empty mbarriers;
//   * warp 1 allocates all 512 TMEM columns (accumulator 0 = block 0 and
//     accumulator 1 = block 1, 128x256 f32 each) and one elected lane issues
//     tcgen05.mma M=128 N=256 K=16 into each accumulator, committing SMEM
//     stages back to the producer and finished accumulators to the epilogue;
//   * warps 2-5 drain accumulator 0 and warps 6-9 accumulator 1 (thread =
//     row): tcgen05.ld, SiLU*up or bf16 cast, all into registers, then the
//     TMEM is released at once so the next tile's MMAs start while the rows
//     go out through a swizzled SMEM box and TMA stores;
//   * tile order: expert by expert; inside an expert, groups of GROUP_PAIRS
//     pairs, all column tiles of a group before the next group, so the
//     group's A rows stay in L2 while every B tile of the expert streams by.
// Every wait is bounded; on a timeout the kernel records it in the status
// word, the roles stop, in-flight copies and MMAs are drained (bounded) and
// TMEM is freed before exit.
#include <cstdint>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BM = 128;                          // rows per block
constexpr int BK = 32;                           // K per pipeline stage
constexpr int BN = 256;                          // MMA N
constexpr int STAGES = 6;
constexpr int GROUP_PAIRS = 4;                   // L2 grouping of pairs inside an expert
constexpr int A_BLOCK_BYTES = BM * BK * 2;       // 8 KB: 128 rows x 64 B (64-byte swizzle)
constexpr int B_BOX_BYTES = BK * 64 * 2;         // 4 KB: 32 k-rows x 64 columns (128-byte swizzle)
constexpr int B_STAGE_BYTES = 4 * B_BOX_BYTES;   // 16 KB
constexpr int STAGE_BYTES = 2 * A_BLOCK_BYTES + B_STAGE_BYTES;  // 32 KB
constexpr int EPI_BOX_BYTES = BM * 64 * 2;       // 16 KB: 128 rows x 64 columns bf16
constexpr int NUM_EPI_GROUPS = 2;
constexpr int EPI_THREADS = 128;                 // per group
constexpr int NUM_THREADS = 64 + NUM_EPI_GROUPS * EPI_THREADS;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;

constexpr int SMEM_STAGE_OFF = 0;
constexpr int SMEM_EPI_OFF = STAGES * STAGE_BYTES;
constexpr int SMEM_BAR_OFF = SMEM_EPI_OFF + NUM_EPI_GROUPS * EPI_BOX_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 1 + 2 + 1;  // full, empty, tmem_full, tmem_empty[2], drain
constexpr int SMEM_PAIR_OFF = SMEM_BAR_OFF + NUM_BARS * 8 + 16;
constexpr int MAX_E = 256;
constexpr int SMEM_BYTES = SMEM_PAIR_OFF + (MAX_E + 1) * 4;
constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;   // slack to align the base to 1024 B

static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

constexpr uint32_t kIdesc = idesc_bf16_f32(128, 256, /*b_mn_major=*/true);

// OR-vote over the 128 threads of epilogue group g (named barrier 2 + 2g).
__device__ __forceinline__ bool vote_any_group(bool flag, int g) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(flag ? 1u : 0u), "r"(2 + 2 * g)
      : "memory");
  return r != 0;
}

struct TileCoord {
  int b0;     // first block of the pair
  int j;      // column tile
  int e;      // expert
  bool two;   // second block b0 + 1 present
  bool ok;
};

// Tile t of the order: expert e (pairs p_off[e] .. p_off[e+1]), then groups
// of GROUP_PAIRS pairs, then column tile, then the pair inside the group.
__device__ __forceinline__ TileCoord decode_tile(int tile, int NT, int E, int num_blocks,
                                                 const int32_t* s_pair_off, const int32_t* __restrict__ off_pad) {
  TileCoord c{0, 0, 0, false, false};
  const int q = tile / NT;  // pair_off[e] <= q < pair_off[e+1]
  int lo = 0, hi = E;       // last e with s_pair_off[e] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pair_off[mid] <= q) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  if (e >= E) return c;
  const int np = s_pair_off[e + 1] - s_pair_off[e];
  const int local = tile - NT * s_pair_off[e];
  if (np <= 0 || local < 0 || local >= NT * np) return c;
  const int g = local / (NT * GROUP_PAIRS);
  const int rem = local - g * NT * GROUP_PAIRS;
  const int gs = min(GROUP_PAIRS, np - g * GROUP_PAIRS);
  const int p = g * GROUP_PAIRS + rem % gs;
  const int blk0 = __ldg(off_pad + e) / BM;
  const int nbe = (__ldg(off_pad + e + 1) - __ldg(off_pad + e)) / BM;
  c.j = rem / gs;
  c.b0 = blk0 + 2 * p;
  c.two = 2 * p + 1 < nbe;
  c.e = e;
  c.ok = c.b0 + (c.two ? 1 : 0) < num_blocks && c.j < NT;
  return c;
}

template <bool kUp>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmD,
                        const int32_t* __restrict__ off_pad, const int32_t* __restrict__ num_blocks_ptr,
                        int max_blocks, int E, int K, int NT, int N_out, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sStage = smem + SMEM_STAGE_OFF;
  uint8_t* sEpi = smem + SMEM_EPI_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SMEM_BAR_OFF);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 1;
  uint64_t* drain = bars + 2 * STAGES + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_pair_off = reinterpret_cast<int32_t*>(smem + SMEM_PAIR_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(&tempty[0], EPI_THREADS);
    mbar_init(&tempty[1], EPI_THREADS);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    prefetch_tmap(&tmB1);
    prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }

  // the prologue above overlaps the previous kernel; from here on this
  // kernel reads what earlier kernels wrote and overwrites what they read
  pdl_wait();
  int num_blocks = __ldg(num_blocks_ptr);
  if (num_blocks > max_blocks || num_blocks < 0) {
    if (threadIdx.x == 0) record_status(status, kStatusBounds);
    num_blocks = num_blocks < 0 ? 0 : max_blocks;
  }
  if (warp == 2) {
    // pairs per expert -> exclusive scan (E <= 256: 8 experts per lane)
    constexpr int per = MAX_E / 32;
    int loc[per];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      int np = 0;
      if (e < E) {
        const int nb = (__ldg(off_pad + e + 1) - __ldg(off_pad + e)) / BM;
        np = nb > 0 ? (nb + 1) / 2 : 0;
      }
      loc[i] = np;
      sum += np;
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
      if (e <= E) s_pair_off[e] = run;  // e == E gets the total (loc of e >= E is 0)
      run += loc[i];
    }
    if (lane == 31 && 32 * per == E) s_pair_off[E] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = NT * s_pair_off[E];
  const int KB = K / BK;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (elect_one_sync()) {
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_normal();
      uint32_t it = 0;  // stages issued so far
      bool stop = false;
      for (int tile = blockIdx.x; tile < total_tiles && !stop; tile += gridDim.x) {
        const TileCoord c = decode_tile(tile, NT, E, num_blocks, s_pair_off, off_pad);
        if (!c.ok) {
          record_status(status, kStatusBounds);
          continue;
        }
        const uint32_t bytes = STAGE_BYTES - (c.two ? 0 : A_BLOCK_BYTES);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, status)) {
            stop = true;
            break;
          }
          uint8_t* st = sStage + s * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], bytes);
          tma_load_2d(st, &tmA, &full[s], kb * BK, c.b0 * BM, pol_a);
          if (c.two) tma_load_2d(st + A_BLOCK_BYTES, &tmA, &full[s], kb * BK, (c.b0 + 1) * BM, pol_a);
          uint8_t* b = st + 2 * A_BLOCK_BYTES;
          const int k0 = c.e * K + kb * BK;
          if (kUp) {
            const int n0 = c.j * 128;
            tma_load_2d(b + 0 * B_BOX_BYTES, &tmB0, &full[s], n0, k0, pol_b);
            tma_load_2d(b + 1 * B_BOX_BYTES, &tmB0, &full[s], n0 + 64, k0, pol_b);
            tma_load_2d(b + 2 * B_BOX_BYTES, &tmB1, &full[s], n0, k0, pol_b);
            tma_load_2d(b + 3 * B_BOX_BYTES, &tmB1, &full[s], n0 + 64, k0, pol_b);
          } else {
            const int n0 = c.j * BN;
#pragma unroll
            for (int q = 0; q < 4; ++q) tma_load_2d(b + q * B_BOX_BYTES, &tmB0, &full[s], n0 + 64 * q, k0, pol_b);
          }
        }
      }
      // drain: every issued stage's copy has landed before the CTA may exit
      const uint32_t nst = it < STAGES ? it : STAGES;
      for (uint32_t s = 0; s < nst; ++s) {
        const uint32_t last = s + STAGES * ((it - 1 - s) / STAGES);
        int no_abort = 0;
        mbar_wait(&full[s], (last / STAGES) & 1u, &no_abort, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (elect_one_sync()) {
      uint32_t it = 0;
      uint32_t tcount = 0;  // tiles processed by this CTA
      bool stop = false;
      for (int tile = blockIdx.x; tile < total_tiles && !stop; tile += gridDim.x) {
        const TileCoord c = decode_tile(tile, NT, E, num_blocks, s_pair_off, off_pad);
        if (!c.ok) continue;
        const uint32_t tph = tcount & 1u;
        // accumulator 0 must be drained before the first MMA; accumulator 1
        // is waited for after the first stage's accumulator-0 MMAs
        if (!mbar_wait(&tempty[0], tph ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, status)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(sStage + s * STAGE_BYTES);
          const uint32_t b_base = st + 2 * A_BLOCK_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major, 64-byte swizzle, 8-row groups 512 B apart; a
            //    16-wide K step is 32 B inside the swizzle atom.
            // B: N-major, 128-byte swizzle; 64-column boxes 4 KB apart
            //    (leading offset), 8-row K groups 1 KB apart (stride
            //    offset); a 16-wide K step is two groups.
            const uint64_t bdesc = smem_desc(b_base + kk * 2048, B_BOX_BYTES, 1024, kSwizzle128B);
            tc_mma_f16(tmem_base, smem_desc(st + kk * 32, 16, 512, kSwizzle64B), bdesc, kIdesc,
                       (kb | kk) != 0 ? 1u : 0u);
          }
          if (kb == 0) {
            if (!mbar_wait(&tempty[1], tph ^ 1u, abort_flag, status)) {
              stop = true;
              break;
            }
            tc_fence_after();
          }
          if (c.two) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t bdesc = smem_desc(b_base + kk * 2048, B_BOX_BYTES, 1024, kSwizzle128B);
              tc_mma_f16(tmem_base + ACC_COLS, smem_desc(st + A_BLOCK_BYTES + kk * 32, 16, 512, kSwizzle64B),
                         bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&empty[s]);
        }
        if (stop) break;
        tc_commit(tfull);
        ++tcount;
      }
      // drain: all issued MMAs complete before TMEM is freed
      tc_commit(drain);
      int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue
    const int g = (warp - 2) >> 2;            // accumulator (= block of the pair) of this group
    const int et = (threadIdx.x - 64) & 127;  // thread index inside the group
    const int q = warp & 3;                   // TMEM lane quarter of this warp
    const int r = q * 32 + lane;              // row of the block owned by this thread
    const uint32_t sync_id = 1 + 2 * g;
    uint8_t* buf = sEpi + g * EPI_BOX_BYTES;
    uint32_t tcount = 0;
    constexpr int NPACK = kUp ? 64 : 128;     // packed bf16 pairs per row of the tile
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const TileCoord c = decode_tile(tile, NT, E, num_blocks, s_pair_off, off_pad);
      if (!c.ok) continue;
      const bool ok = mbar_wait(tfull, tcount & 1u, abort_flag, status);
      if (vote_any_group(!ok, g)) break;
      tc_fence_after();
      const bool mine = (g == 0) || c.two;
      uint32_t packed[NPACK];
      if (mine) {
        const uint32_t tbase = tmem_base + g * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
        if (kUp) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t gv[32], uv[32];
            tmem_ld_32x32b_x32(tbase + ch * 32, gv);
            tmem_ld_32x32b_x32(tbase + 128 + ch * 32, uv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(gv[2 * i]), g1 = __uint_as_float(gv[2 * i + 1]);
              const float u0 = __uint_as_float(uv[2 * i]), u1 = __uint_as_float(uv[2 * i + 1]);
              // silu(g) = g * sigmoid(g); exp and reciprocal at the SFU's
              // approximate precision (a few float32 ulps, far below the
              // bf16 rounding of h).  For g < -88, exp(-g) = inf and the
              // reciprocal gives 0, the limit of sigmoid.
              const float h0 = g0 * __fdividef(1.0f, 1.0f + __expf(-g0)) * u0;
              const float h1 = g1 * __fdividef(1.0f, 1.0f + __expf(-g1)) * u1;
              packed[ch * 16 + i] = pack_bf16x2(h0, h1);
            }
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + ch * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[ch * 16 + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          }
        }
      }
      // the accumulator is in registers: release TMEM to the next tile's MMAs
      tc_fence_before();
      mbar_arrive(&tempty[g]);
      ++tcount;
      if (!mine) continue;
      const int row0 = (c.b0 + g) * BM;
      constexpr int NBOX = kUp ? 2 : 4;  // 64-column output boxes
#pragma unroll
      for (int bx = 0; bx < NBOX; ++bx) {
        if (et == 0) tma_store_wait_read<0>();  // the box's previous store has read `buf`
        named_barrier_sync(sync_id, EPI_THREADS);
        // 128-byte swizzle: logical 16-B chunk cidx of row r sits at cidx ^ (r % 8)
        uint8_t* row_ptr = buf + r * 128;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint32_t* src = packed + bx * 32 + 4 * m;
          *reinterpret_cast<uint4*>(row_ptr + ((m ^ (r & 7)) << 4)) = make_uint4(src[0], src[1], src[2], src[3]);
        }
        fence_proxy_async_smem();
        named_barrier_sync(sync_id, EPI_THREADS);
        if (et == 0) {
          const int col0 = (kUp ? c.j * 128 : c.j * BN) + bx * 64;
          if (col0 < N_out) tma_store_2d(&tmD, buf, col0, row0);  // no store wholly past the last column
          tma_store_commit();
        }
      }
    }
    if (et == 0) tma_store_wait_all<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

__global__ void permute_rows_kernel(const uint16_t* __restrict__ X, const int32_t* __restrict__ gather_idx,
                                    const int32_t* __restrict__ num_blocks_ptr, int64_t max_rows, int T, int H,
                                    uint16_t* __restrict__ Xp, uint32_t* __restrict__ status) {
  pdl_launch_dependents();
  pdl_wait();
  int64_t rows = static_cast<int64_t>(__ldg(num_blocks_ptr)) * BM;
  if (rows > max_rows || rows < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_status(status, kStatusBounds);
    rows = rows < 0 ? 0 : max_rows;
  }
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int vec_per_row = H / 8;
  for (int64_t row = warp0; row < rows; row += nwarps) {
    const int t = __ldg(gather_idx + row);
    if (t < 0) continue;
    if (t >= T) {
      if (lane == 0) record_status(status, kStatusBounds);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(Xp + row * H);
#pragma unroll 4
    for (int v = lane; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
  }
}

template <bool kUp>
cudaError_t launch_gemm(const moe_shape& s, const GemmMaps& maps, const int32_t* off_pad,
                        const int32_t* block_expert, const int32_t* num_blocks, uint32_t* status, int num_sms,
                        cudaStream_t st) {
  (void)block_expert;  // tiles are decoded from off_pad
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !attr_done[dev]) {
    err = cudaFuncSetAttribute(grouped_gemm_kernel<kUp>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (err != cudaSuccess) return err;
    attr_done[dev] = true;
  }
  // up: 128 gate + 128 up columns per tile (I % 128 == 0); down: 256 output
  // columns per tile, the last tile of an H % 256 == 128 row is half outside
  // the tensor (TMA zero-fills those weight columns and skips the store).
  const int NT = kUp ? s.I / 128 : (s.H + BN - 1) / BN;
  const int K = kUp ? s.H : s.I;
  const int64_t mb = max_blocks_of(s);
  const int64_t max_tiles = (mb / 2 + s.E) * NT;  // sum_e ceil(nb_e / 2) <= nb / 2 + E
  const int grid = static_cast<int>(max_tiles < num_sms ? max_tiles : num_sms);
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(grouped_gemm_kernel<kUp>, dim3(grid), dim3(NUM_THREADS), SMEM_ALLOC, st, maps.a, maps.b0,
                    maps.b1, maps.d, off_pad, num_blocks, static_cast<int>(mb), s.E, K, NT, kUp ? s.I : s.H,
                    status);
}

}  // namespace

cudaError_t launch_permute_rows(const moe_shape& s, const uint16_t* X, const int32_t* gather_idx,
                                const int32_t* num_blocks, uint16_t* Xp, uint32_t* status, cudaStream_t st) {
  const int64_t mr = max_rows_of(s);
  const int threads = 256;
  int64_t blocks = (mr + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(permute_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st, X, gather_idx,
                    num_blocks, mr, s.T, s.H, Xp, status);
}

cudaError_t launch_gemm_up(const moe_shape& s, const GemmMaps& maps, const int32_t* off_pad,
                           const int32_t* block_expert, const int32_t* num_blocks, uint32_t* status, int num_sms,
                           cudaStream_t st) {
  return launch_gemm<true>(s, maps, off_pad, block_expert, num_blocks, status, num_sms, st);
}

cudaError_t launch_gemm_down(const moe_shape& s, const GemmMaps& maps, const int32_t* off_pad,
                             const int32_t* block_expert, const int32_t* num_blocks, uint32_t* status, int num_sms,
                             cudaStream_t st) {
  return launch_gemm<false>(s, maps, off_pad, block_expert, num_blocks, status, num_sms, st);
}

}  // namespace moe
