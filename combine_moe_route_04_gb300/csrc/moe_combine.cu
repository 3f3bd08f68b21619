// moe_combine.cu -- top-k weighted combine back to token order.
//
// What it computes ("通算融合算子（一）：为什么要把通信写进 GEMM kernel 里" §4, table of
// data-flow patterns, "GEMM + combine": the top-k weighted reduction):
//   out[t, c] = bf16( sum_{j = 0..k-1} w[t, j] * Y[scatter_idx[t, j], c] )
// with a float32 accumulator in slot order, each product and each sum rounded
// to float32 (__fmul_rn / __fadd_rn keep the compiler from fusing them).
//
// One thread per 8 output columns of one token: it gathers the k expert rows
// of its token with 16-byte loads (all k loads issued before the sums, for
// memory-level parallelism), so a warp reads 512 contiguous bytes of each
// expert row and writes 512 contiguous bytes of out.  No atomics: results are
// bitwise reproducible.
#include <cstdint>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kMaxK = 16;

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ Y,
                                                      const int32_t* __restrict__ scatter_idx,
                                                      const float* __restrict__ topk_w, int T, int H, int k,
                                                      int64_t max_rows, uint16_t* __restrict__ out,
                                                      uint32_t* __restrict__ status) {
  const int vec_per_row = H / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(T) * vec_per_row) return;
  const int t = static_cast<int>(idx / vec_per_row);
  const int v = static_cast<int>(idx - static_cast<int64_t>(t) * vec_per_row);

  int64_t rows[kMaxK];
  float w[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    rows[j] = -1;
    w[j] = 0.0f;
    if (j < k) {
      const int64_t r = __ldg(scatter_idx + static_cast<int64_t>(t) * k + j);
      w[j] = __ldg(topk_w + static_cast<int64_t>(t) * k + j);
      if (r >= 0 && r < max_rows) {
        rows[j] = r;
      } else if (status != nullptr) {
        record_status(status, kStatusBounds);
      }
    }
  }
  uint4 y[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    y[j] = make_uint4(0u, 0u, 0u, 0u);
    if (j < k && rows[j] >= 0) y[j] = __ldg(reinterpret_cast<const uint4*>(Y + rows[j] * H) + v);
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k) {
      const uint32_t p[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w[j], bf16lo_to_f32(p[i])));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w[j], bf16hi_to_f32(p[i])));
      }
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H)[v] = o;
}

}  // namespace

cudaError_t launch_combine(const moe_shape& s, const uint16_t* Y, const int32_t* scatter_idx, const float* topk_w,
                           uint16_t* out, uint32_t* status, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(s.T) * (s.H / 8);
  const int threads = 256;
  combine_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, st>>>(
      Y, scatter_idx, topk_w, s.T, s.H, s.k, max_rows_of(s), out, status);
  return cudaGetLastError();
}

}  // namespace moe
