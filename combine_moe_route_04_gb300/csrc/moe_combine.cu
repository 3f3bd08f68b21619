// moe_combine.cu -- top-k weighted combine back to token order.
//
// What it computes ("通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §4, table of
// data-flow patterns, "GEMM + combine": the top-k weighted reduction):
//   out[t, c] = bf16( sum_{j = 0..k-1} w[t, j] * Y[scatter_idx[t, j], c] )
// with a float32 accumulator in slot order, each product and each sum rounded
// to float32 (__fmul_rn / __fadd_rn keep the compiler from fusing them).
//
// One warp per token, or per piece of a token when there are fewer tokens
// than resident warps (decode): a warp reads 512 contiguous bytes of each of
// the k expert rows per load instruction and writes 512 contiguous bytes of
// out.  (Measured: pieces for every shape cost the large workloads 1.5%; one
// warp per token left decode's 64 tokens on 8 SMs, 13 us slower.)
// No atomics: results are bitwise reproducible.
#include <cstdint>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

// One warp per work item (grid-stride), an item being one of a token's ppt
// pieces (ppt = 1: the whole token): lanes j < k load the token's row index
// and weight and broadcast them; then per iteration each lane gathers CH
// 16-byte chunks of all k expert rows (k*CH loads in flight per lane) and sums
// them in slot order.
template <int KMAX, int CH>
__global__ void __launch_bounds__(256, 2) combine_kernel(const uint16_t* __restrict__ Y,
                                                      const int32_t* __restrict__ scatter_idx,
                                                      const float* __restrict__ topk_w, int T, int H, int k,
                                                      int64_t max_rows, int ppt, uint16_t* __restrict__ out,
                                                      uint32_t* __restrict__ status) {
  pdl_wait();
  // the next kernel (the next forward's routing) may launch only now, so its
  // CTAs do not wait on SMs through the down GEMM this kernel waited for
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int vpr = H / 8;  // 16-byte chunks per row
  const int iters = (vpr + 32 * CH - 1) / (32 * CH);  // iterations per row
  const int per = (iters + ppt - 1) / ppt;              // iterations per piece
  const int64_t items = static_cast<int64_t>(T) * ppt;
  for (int64_t item = warp0; item < items; item += nwarps) {
    const int64_t t = item / ppt;
    const int first = static_cast<int>(item % ppt) * per * 32 * CH;
    const int last = min(vpr, first + per * 32 * CH);
    int my_row = -1;
    float my_w = 0.0f;
    if (lane < k) {
      const int64_t r = __ldg(scatter_idx + t * k + lane);
      my_w = __ldg(topk_w + t * k + lane);
      if (r >= 0 && r < max_rows) {
        my_row = static_cast<int>(r);
      } else if (status != nullptr && first == 0) {
        record_status(status, kStatusBounds);
      }
    }
    int rows[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      rows[j] = __shfl_sync(0xffffffffu, my_row, j);
      w[j] = __shfl_sync(0xffffffffu, my_w, j);
    }
    const uint4* Y4 = reinterpret_cast<const uint4*>(Y);
    uint4* orow = reinterpret_cast<uint4*>(out + t * H);
    for (int c0 = first; c0 < last; c0 += 32 * CH) {
      uint4 y[KMAX][CH];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
#pragma unroll
        for (int cc = 0; cc < CH; ++cc) {
          const int v = c0 + cc * 32 + lane;
          y[j][cc] = make_uint4(0u, 0u, 0u, 0u);
          if (j < k && rows[j] >= 0 && v < vpr) y[j][cc] = __ldg(Y4 + static_cast<int64_t>(rows[j]) * vpr + v);
        }
      }
#pragma unroll
      for (int cc = 0; cc < CH; ++cc) {
        const int v = c0 + cc * 32 + lane;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (j < k) {
            const uint32_t p[4] = {y[j][cc].x, y[j][cc].y, y[j][cc].z, y[j][cc].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w[j], bf16lo_to_f32(p[i])));
              acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w[j], bf16hi_to_f32(p[i])));
            }
          }
        }
        if (v < vpr) {
          uint4 o;
          o.x = pack_bf16x2(acc[0], acc[1]);
          o.y = pack_bf16x2(acc[2], acc[3]);
          o.z = pack_bf16x2(acc[4], acc[5]);
          o.w = pack_bf16x2(acc[6], acc[7]);
          orow[v] = o;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine(const moe_shape& s, const uint16_t* Y, const int32_t* scatter_idx, const float* topk_w,
                           uint16_t* out, uint32_t* status, int num_sms, cudaStream_t st) {
  // pieces per token: enough for the items to fill the resident warps (2
  // CTAs of 8 warps per SM), rounded up, at most one per iteration of the
  // row (measured: 2048 tokens in 2 pieces, 512 CTAs, forward 1.3% faster
  // than 1 piece, 256 CTAs spread unevenly over the SMs)
  const int64_t vpr = s.H / 8;
  const int64_t iters = s.k <= 8 ? (vpr + 63) / 64 : (vpr + 31) / 32;
  int64_t ppt = (static_cast<int64_t>(num_sms) * 16 + s.T - 1) / s.T;
  if (ppt < 1) ppt = 1;
  if (ppt > iters) ppt = iters;
  int64_t blocks = (static_cast<int64_t>(s.T) * ppt + 7) / 8;  // 8 warps (items) per CTA
  if (blocks > 4096) blocks = 4096;
  const int64_t mr = max_rows_of(s);
  if (s.k <= 8)
    return launch_pdl(combine_kernel<8, 2>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, Y, scatter_idx,
                      topk_w, s.T, s.H, s.k, mr, static_cast<int>(ppt), out, status);
  return launch_pdl(combine_kernel<16, 1>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, Y, scatter_idx,
                    topk_w, s.T, s.H, s.k, mr, static_cast<int>(ppt), out, status);
}

}  // namespace moe
