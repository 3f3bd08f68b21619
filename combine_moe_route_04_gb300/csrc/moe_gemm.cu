// moe_gemm.cu -- persistent, warp-specialised grouped GEMMs of the expert
// layer on the sm_103a tensor cores (tcgen05 + TMEM + TMA), and the row
// gather that feeds the gate/up GEMM.
//
// What they compute ("通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §1: gate/up
// GEMM -> SiLU -> down GEMM; "通算融合算子（三）：ThunderKittens 多卡编程与可融合的
// GEMM 模板" §4: each 128-row block multiplies the weights of its own expert,
// tasks visited expert-major):
//   up:   for each 128-row block b of expert e and each 128-column slice j,
//         G = A_b Wg[e][:, j], U = A_b Wu[e][:, j]  (float32 in TMEM)
//         h[b, j] = bf16(silu(G) * U)
//   down: Y[b, j] = bf16(h_b Wd[e][:, j]) for 256-column slices j.
//
// Design (the pipeline roles and barrier lifetimes of "TIRx 与高性能GEMM (下)"
// Step 7, re-keyed to expert blocks):
//   warp 0  TMA producer: A tile 128x64 (K-major) and B tile 64x256 (N-major,
//           four 64x64 boxes) per stage into a 4-stage SMEM ring, 128-byte
//           swizzle, completion counted on full[s];
//   warp 1  allocates 512 TMEM columns (two 128x256 f32 accumulators) and one
//           elected lane issues tcgen05.mma (M=128, N=256, K=16) per 16-wide
//           K step; tcgen05.commit frees SMEM stages (empty[s]) and publishes
//           a finished accumulator (tmem_full[a]);
//   warps 2-5 (128 threads) epilogue: tcgen05.ld the accumulator (thread =
//           row), release it (tmem_empty[a]) so the MMA of the next tile
//           overlaps this writeback, apply SiLU*up / bf16 cast, write a
//           swizzled 128x64 SMEM tile and TMA-store it (double-buffered).
//   Tiles are visited expert by expert, column slice by column slice, block
//   by block, so CTAs running at the same time share weight tiles in L2.
//   Every wait is bounded; on a timeout the kernel records it in the status
//   word, the roles stop, in-flight copies and MMAs are drained (bounded) and
//   TMEM is freed before exit.
#include <cstdint>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BM = 128;                         // rows per tile (one expert block)
constexpr int BK = 64;                          // K per pipeline stage (128 B of bf16)
constexpr int BN = 256;                         // MMA N
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BOX_BYTES = BK * 64 * 2;        // 8 KB: 64 k-rows x 64 columns
constexpr int B_STAGE_BYTES = 4 * B_BOX_BYTES;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int EPI_BOX_BYTES = BM * 64 * 2;      // 16 KB: 128 rows x 64 columns bf16
constexpr int EPI_BUFS = 2;
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;

constexpr int SMEM_A_OFF = 0;
constexpr int SMEM_B_OFF = SMEM_A_OFF + STAGES * A_STAGE_BYTES;
constexpr int SMEM_EPI_OFF = SMEM_B_OFF + STAGES * B_STAGE_BYTES;
constexpr int SMEM_BAR_OFF = SMEM_EPI_OFF + EPI_BUFS * EPI_BOX_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
constexpr int SMEM_BYTES = SMEM_BAR_OFF + NUM_BARS * 8 + 16;
constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;   // slack to align the base to 1024 B

static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

constexpr uint32_t kIdesc = idesc_bf16_f32(128, 256, /*b_mn_major=*/true);

__device__ __forceinline__ bool vote_any_epi(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 2, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(flag ? 1u : 0u)
      : "memory");
  return r != 0;
}

struct TileCoord {
  int b;      // 128-row block
  int j;      // column slice
  int e;      // expert
  bool ok;
};

// Tile order: expert-major, then column slice, then the expert's blocks.
// tile / NT falls inside the expert's blocks, so block_expert[tile / NT]
// names the expert without a search.
__device__ __forceinline__ TileCoord decode_tile(int tile, int NT, int num_blocks, int E,
                                                 const int32_t* __restrict__ off_pad,
                                                 const int32_t* __restrict__ block_expert) {
  TileCoord c{0, 0, 0, false};
  const int bq = tile / NT;
  const int e = __ldg(block_expert + bq);
  if (e < 0 || e >= E) return c;
  const int blk0 = __ldg(off_pad + e) / BM;
  const int nbe = (__ldg(off_pad + e + 1) - __ldg(off_pad + e)) / BM;
  if (nbe <= 0 || blk0 < 0 || blk0 + nbe > num_blocks) return c;
  const int local = tile - NT * blk0;
  if (local < 0 || local >= NT * nbe) return c;
  c.j = local / nbe;
  c.b = blk0 + local % nbe;
  c.e = e;
  c.ok = true;
  return c;
}

template <bool kUp>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmD,
                        const int32_t* __restrict__ off_pad, const int32_t* __restrict__ block_expert,
                        const int32_t* __restrict__ num_blocks_ptr, int max_blocks, int E, int K, int NT,
                        int N_out, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + SMEM_A_OFF;
  uint8_t* sB = smem + SMEM_B_OFF;
  uint8_t* sEpi = smem + SMEM_EPI_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SMEM_BAR_OFF);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], EPI_THREADS);
    }
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // the prologue above overlaps the previous kernel; from here on this
  // kernel reads what earlier kernels wrote and overwrites what they read
  pdl_wait();
  int num_blocks = __ldg(num_blocks_ptr);
  if (num_blocks > max_blocks || num_blocks < 0) {
    if (threadIdx.x == 0) record_status(status, kStatusBounds);
    num_blocks = num_blocks < 0 ? 0 : max_blocks;
  }
  const int total_tiles = num_blocks * NT;
  const int KB = K / BK;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (elect_one_sync()) {
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_normal();
      uint32_t it = 0;  // stages issued so far
      bool stop = false;
      for (int tile = blockIdx.x; tile < total_tiles && !stop; tile += gridDim.x) {
        const TileCoord c = decode_tile(tile, NT, num_blocks, E, off_pad, block_expert);
        if (!c.ok) {
          record_status(status, kStatusBounds);
          continue;
        }
        const int brow = c.e * K;  // first weight row of the expert
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, status)) {
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          tma_load_2d(sA + s * A_STAGE_BYTES, &tmA, &full[s], kb * BK, c.b * BM, pol_a);
          uint8_t* b = sB + s * B_STAGE_BYTES;
          const int k0 = brow + kb * BK;
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
        const TileCoord c = decode_tile(tile, NT, num_blocks, E, off_pad, block_expert);
        if (!c.ok) continue;
        const uint32_t a = tcount & 1u;
        const uint32_t aph = (tcount >> 1) & 1u;
        if (!mbar_wait(&tempty[a], aph ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + a * ACC_COLS;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, status)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + s * A_STAGE_BYTES);
          const uint32_t b_base = smem_u32(sB + s * B_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major, 128-B swizzle, 8-row groups 1024 B apart; a 16-wide
            //    K step is 32 B inside the swizzle atom.
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            // B: N-major, 128-B swizzle; 64-column boxes 8 KB apart (leading
            //    offset), 8-row K groups 1024 B apart (stride offset); a
            //    16-wide K step is two groups.
            const uint64_t bdesc = smem_desc_sw128(b_base + kk * 2048, B_BOX_BYTES, 1024);
            tc_mma_f16(d, adesc, bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        if (stop) break;
        tc_commit(&tfull[a]);
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
    const int et = threadIdx.x - 64;          // 0..127
    const int q = warp & 3;                   // TMEM lane quarter of this warp
    const int r = q * 32 + lane;              // row of the tile owned by this thread
    uint32_t tcount = 0;
    uint32_t nstore = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const TileCoord c = decode_tile(tile, NT, num_blocks, E, off_pad, block_expert);
      if (!c.ok) continue;
      const uint32_t a = tcount & 1u;
      const uint32_t aph = (tcount >> 1) & 1u;
      const bool ok = mbar_wait(&tfull[a], aph, abort_flag, status);
      if (vote_any_epi(!ok)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + a * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      constexpr int NCHUNK = kUp ? 2 : 4;  // 64-column output boxes per tile
#pragma unroll 1
      for (int ch = 0; ch < NCHUNK; ++ch) {
        uint8_t* buf = sEpi + (nstore & 1u) * EPI_BOX_BYTES;
        if (et == 0) tma_store_wait_read<1>();  // the store that last read `buf` is done
        named_barrier_sync(1, EPI_THREADS);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t col = ch * 64 + half * 32;
          uint32_t packed[16];
          if (kUp) {
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(tbase + col, g);
            tmem_ld_32x32b_x32(tbase + 128 + col, u);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
              const float h0 = g0 / (1.0f + __expf(-g0)) * u0;
              const float h1 = g1 / (1.0f + __expf(-g1)) * u1;
              packed[i] = pack_bf16x2(h0, h1);
            }
          } else {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + col, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          }
          // 128-B swizzle: logical 16-B chunk cidx of row r sits at cidx ^ (r % 8)
          uint8_t* row_ptr = buf + r * 128;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int cidx = half * 4 + m;
            uint4 v4 = make_uint4(packed[4 * m], packed[4 * m + 1], packed[4 * m + 2], packed[4 * m + 3]);
            *reinterpret_cast<uint4*>(row_ptr + ((cidx ^ (r & 7)) << 4)) = v4;
          }
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, EPI_THREADS);
        if (et == 0) {
          const int col0 = kUp ? c.j * 128 + ch * 64 : c.j * BN + ch * 64;
          if (col0 < N_out) tma_store_2d(&tmD, buf, col0, c.b * BM);  // no store wholly past the last column
          tma_store_commit();
        }
        ++nstore;
      }
      tc_fence_before();
      mbar_arrive(&tempty[a]);
      ++tcount;
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
  // the tensor (TMA zero-fills those weight columns and clips the store).
  const int NT = kUp ? s.I / 128 : (s.H + BN - 1) / BN;
  const int K = kUp ? s.H : s.I;
  const int64_t mb = max_blocks_of(s);
  const int64_t max_tiles = mb * NT;
  const int grid = static_cast<int>(max_tiles < num_sms ? max_tiles : num_sms);
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(grouped_gemm_kernel<kUp>, dim3(grid), dim3(NUM_THREADS), SMEM_ALLOC, st, maps.a, maps.b0,
                    maps.b1, maps.d, off_pad, block_expert, num_blocks, static_cast<int>(mb), s.E, K, NT,
                    kUp ? s.I : s.H, status);
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
