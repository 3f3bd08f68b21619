// moe_api.cu -- the C ABI declared in include/moe.h: argument and shape
// validation, device checks, workspace layout, TMA tensor-map encoding and the
// launch sequence of each step.  Host code only; it allocates no device memory.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "moe_internal.h"

namespace moe {
namespace {

struct DevInfo {
  bool valid = false;
  bool arch_ok = false;
  int num_sms = 0;
};

DevInfo g_dev[64];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

constexpr size_t kAlign = 1024;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_shape(const moe_shape* s) {
  if (s == nullptr) return MOE_ERR_INVALID_ARG;
  if (s->T < 1 || s->T > (1 << 22)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->E < 1 || s->E > 256) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->k < 1 || s->k > 16 || s->k > s->E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->H < 128 || s->H > 32768 || s->H % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->I < 128 || s->I > 32768 || s->I % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

// Makes the stream's device current for this library's launches (the
// previous current device goes into `restore`, which puts it back when the
// entry point returns) and checks it is a compute capability 10.3 part.
moe_status prepare_device(cudaStream_t st, int* num_sms, DeviceRestore* restore) {
  int dev = 0;
  cudaError_t err;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (st != nullptr && cudaStreamIsCapturing(st, &cs) != cudaSuccess) return MOE_ERR_CUDA;
  if (st != nullptr && cs == cudaStreamCaptureStatusNone) {
    err = cudaStreamGetDevice(st, &dev);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return MOE_ERR_CUDA;
    if (cur != dev) {
      if (cudaSetDevice(dev) != cudaSuccess) return MOE_ERR_CUDA;
      if (restore != nullptr && restore->prev < 0) restore->prev = cur;
    }
  } else if (cudaGetDevice(&dev) != cudaSuccess) {  // no stream, or a stream being captured (its device is current)
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.valid) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.arch_ok = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.valid = true;
  }
  if (!d.arch_ok) return MOE_ERR_ARCH;
  if (num_sms) *num_sms = d.num_sms;
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return MOE_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return MOE_OK;
}

struct Views {
  uint32_t* status;
  int32_t* chunk_counts;
  uint16_t* xp;
  uint32_t* win_done;
  int32_t* local_rank;
  moe_views v;
};

Views views_of(const moe_shape& s, void* ws) {
  const WsLayout L = ws_layout(s);
  uint8_t* b = static_cast<uint8_t*>(ws);
  Views w;
  w.status = reinterpret_cast<uint32_t*>(b + L.status);
  w.chunk_counts = reinterpret_cast<int32_t*>(b + L.chunk_counts);
  w.xp = reinterpret_cast<uint16_t*>(b + L.xp);
  w.win_done = reinterpret_cast<uint32_t*>(b + L.win_done);
  w.local_rank = reinterpret_cast<int32_t*>(b + L.local_rank);
  w.v.Xp = reinterpret_cast<moe_bf16*>(w.xp);
  w.v.topk_ids = reinterpret_cast<int32_t*>(b + L.topk_ids);
  w.v.topk_w = reinterpret_cast<float*>(b + L.topk_w);
  w.v.counts = reinterpret_cast<int32_t*>(b + L.counts);
  w.v.off_pad = reinterpret_cast<int32_t*>(b + L.off_pad);
  w.v.block_expert = reinterpret_cast<int32_t*>(b + L.block_expert);
  w.v.num_blocks = reinterpret_cast<int32_t*>(b + L.num_blocks);
  w.v.gather_idx = reinterpret_cast<int32_t*>(b + L.gather_idx);
  w.v.scatter_idx = reinterpret_cast<int32_t*>(b + L.scatter_idx);
  w.v.h = reinterpret_cast<moe_bf16*>(b + L.h);
  w.v.Y = reinterpret_cast<moe_bf16*>(b + L.y);
  return w;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The gate/up GEMM over rows already in expert order (Xp [max_rows][H]).
// win_done: nullptr, or the forward's per-window counters (see launch_gemm_up).
moe_status run_up_rows(const moe_shape& s, const uint16_t* Xp, const int32_t* counts, const int32_t* off_pad,
                       const uint16_t* Wg, const uint16_t* Wu, uint16_t* h, const Views& w, uint32_t* win_done,
                       int num_sms, cudaStream_t st) {
  const uint64_t mr = static_cast<uint64_t>(max_rows_of(s));
  GemmMaps m;
  const uint64_t EH = static_cast<uint64_t>(s.E) * s.H;
  if (!encode_bf16_2d(&m.a, Xp, mr, s.H, 128, 32) || !encode_bf16_2d(&m.b0, Wg, EH, s.I, 32, 64) ||
      !encode_bf16_2d(&m.b1, Wu, EH, s.I, 32, 64) || !encode_bf16_2d(&m.a64, Xp, mr, s.H, 64, 32) ||
      !encode_bf16_2d(&m.a80, Xp, mr, s.H, 80, 32))
    return MOE_ERR_CUDA;
  return cuda_status(
      launch_gemm_up(s, m, h, off_pad, counts, w.status, ws_sched_up(w.status), win_done, num_sms, st));
}

// Row gather into the workspace's Xp (token by token: each row of X read
// once), then the GEMM over it, which starts when the gather has completed.
// win_done: nullptr, or the forward's per-window counters.
moe_status run_up(const moe_shape& s, const uint16_t* X, const int32_t* scatter_idx, const int32_t* counts,
                  const int32_t* off_pad, const uint16_t* Wg, const uint16_t* Wu,
                  uint16_t* h, const Views& w, uint32_t* win_done, int num_sms, cudaStream_t st) {
  cudaError_t e = launch_scatter_rows(s, X, scatter_idx, w.xp, w.status, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return run_up_rows(s, w.xp, counts, off_pad, Wg, Wu, h, w, win_done, num_sms, st);
}

moe_status run_down(const moe_shape& s, const uint16_t* h, const int32_t* counts, const int32_t* off_pad,
                    const uint16_t* Wd, uint16_t* Y, const Views& w, uint32_t* win_done, int num_sms,
                    cudaStream_t st) {
  const uint64_t mr = static_cast<uint64_t>(max_rows_of(s));
  GemmMaps m;
  const uint64_t EI = static_cast<uint64_t>(s.E) * s.I;
  if (!encode_bf16_2d(&m.a, h, mr, s.I, 128, 32) || !encode_bf16_2d(&m.b0, Wd, EI, s.H, 32, 64) ||
      !encode_bf16_2d(&m.a64, h, mr, s.I, 64, 32) || !encode_bf16_2d(&m.a80, h, mr, s.I, 80, 32))
    return MOE_ERR_CUDA;
  m.b1 = m.b0;
  return cuda_status(
      launch_gemm_down(s, m, Y, off_pad, counts, w.status, ws_sched_down(w.status), win_done, num_sms, st));
}

}  // namespace

moe_status device_ready(cudaStream_t st, int* num_sms, DeviceRestore* restore) {
  return prepare_device(st, num_sms, restore);
}
moe_status validate_shape(const moe_shape* s) { return check_shape(s); }

WsLayout ws_layout(const moe_shape& s) {
  WsLayout L{};
  const size_t T = static_cast<size_t>(s.T), E = static_cast<size_t>(s.E), k = static_cast<size_t>(s.k);
  const size_t mr = static_cast<size_t>(max_rows_of(s));
  const size_t mb = static_cast<size_t>(max_blocks_of(s));
  const size_t nch = static_cast<size_t>(num_chunks_of(s));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  L.status = take(256);
  L.chunk_counts = take(E * nch * 4);
  L.xp = take(mr * static_cast<size_t>(s.H) * 2);
  L.topk_ids = take(T * k * 4);
  L.topk_w = take(T * k * 4);
  L.counts = take(E * 4);
  L.off_pad = take((E + 1) * 4);
  L.block_expert = take(mb * 4);
  L.num_blocks = take(4);
  L.gather_idx = take(mr * 4);
  L.scatter_idx = take(T * k * 4);
  L.local_rank = take(T * k * 4);
  L.h = take(mr * static_cast<size_t>(s.I) * 2);
  L.y = take(mr * static_cast<size_t>(s.H) * 2);
  L.win_done = take(static_cast<size_t>(forward_counters_of(s)) * 4);
  L.total = off;
  return L;
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_cols) {
  if (g_encode == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_cols * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_cols * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                     : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    case MOE_ERR_ARCH: return "MOE_ERR_ARCH";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
    case MOE_ERR_SCRATCH_LIMIT: return "MOE_ERR_SCRATCH_LIMIT";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_capacity(const moe_shape* shape, int64_t* max_blocks, int64_t* max_rows) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (max_blocks == nullptr || max_rows == nullptr) return MOE_ERR_INVALID_ARG;
  *max_blocks = max_blocks_of(*shape);
  *max_rows = max_rows_of(*shape);
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(*shape).total;
  return MOE_OK;
}

moe_status moe_workspace_views(const moe_shape* shape, void* ws, moe_views* views) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (ws == nullptr || views == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  *views = views_of(*shape, ws).v;
  return MOE_OK;
}

moe_status moe_workspace_init(const moe_shape* shape, void* ws, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceRestore restore;
  st = prepare_device(s, nullptr, &restore);
  if (st != MOE_OK) return st;
  return cuda_status(cudaMemsetAsync(ws, 0, 256, s));
}

moe_status moe_last_device_status(void* ws, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceRestore restore;
  moe_status st = prepare_device(s, nullptr, &restore);
  if (st != MOE_OK) return st;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (word != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof word, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (word & kStatusTimeout) return MOE_ERR_TIMEOUT;
  if (word & kStatusBounds) return MOE_ERR_DEVICE_BOUNDS;
  return MOE_OK;
}

moe_status moe_check_wait_timeout(void* ws, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceRestore restore;
  moe_status st = prepare_device(s, nullptr, &restore);
  if (st != MOE_OK) return st;
  return cuda_status(launch_wait_timeout(static_cast<uint32_t*>(ws), s));
}

moe_status moe_route(const moe_shape* shape, const float* logits, int32_t* topk_ids, float* topk_w,
                     int32_t* counts, int32_t* off_pad, int32_t* block_expert, int32_t* num_blocks,
                     int32_t* gather_idx, int32_t* scatter_idx, void* ws, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {logits, topk_ids, topk_w, counts, off_pad, block_expert, num_blocks, gather_idx,
                        scatter_idx, ws};
  for (const void* p : ptrs) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceRestore restore;
  st = prepare_device(s, nullptr, &restore);
  if (st != MOE_OK) return st;
  const Views w = views_of(*shape, ws);
  return cuda_status(launch_route(*shape, logits, topk_ids, topk_w, counts, off_pad, block_expert, num_blocks,
                                  gather_idx, scatter_idx, w.chunk_counts, ws_route_counter(w.status), w.status,
                                  s));
}

moe_status moe_grouped_gemm_up(const moe_shape* shape, const moe_bf16* X, const int32_t* scatter_idx,
                               const int32_t* counts, const int32_t* off_pad, const moe_bf16* W_gate,
                               const moe_bf16* W_up, moe_bf16* h, void* ws, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {X, scatter_idx, counts, off_pad, W_gate, W_up, h, ws};
  for (const void* p : ptrs) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int sms = 0;
  DeviceRestore restore;
  st = prepare_device(s, &sms, &restore);
  if (st != MOE_OK) return st;
  return run_up(*shape, X, scatter_idx, counts, off_pad, W_gate, W_up, h, views_of(*shape, ws), nullptr, sms, s);
}

moe_status moe_grouped_gemm_up_rows(const moe_shape* shape, const moe_bf16* Xp, const int32_t* counts,
                                    const int32_t* off_pad, const moe_bf16* W_gate, const moe_bf16* W_up,
                                    moe_bf16* h, void* ws, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {Xp, counts, off_pad, W_gate, W_up, h, ws};
  for (const void* p : ptrs) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int sms = 0;
  DeviceRestore restore;
  st = prepare_device(s, &sms, &restore);
  if (st != MOE_OK) return st;
  return run_up_rows(*shape, Xp, counts, off_pad, W_gate, W_up, h, views_of(*shape, ws), nullptr, sms, s);
}

moe_status moe_grouped_gemm_down(const moe_shape* shape, const moe_bf16* h, const int32_t* counts,
                                 const int32_t* off_pad, const moe_bf16* W_down, moe_bf16* Y, void* ws,
                                 moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {h, counts, off_pad, W_down, Y, ws};
  for (const void* p : ptrs) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int sms = 0;
  DeviceRestore restore;
  st = prepare_device(s, &sms, &restore);
  if (st != MOE_OK) return st;
  return run_down(*shape, h, counts, off_pad, W_down, Y, views_of(*shape, ws), nullptr, sms, s);
}

moe_status moe_combine(const moe_shape* shape, const moe_bf16* Y, const int32_t* scatter_idx, const float* topk_w,
                       moe_bf16* out, void* ws, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {Y, scatter_idx, topk_w, out};
  for (const void* p : ptrs) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  }
  if (ws != nullptr && !aligned16(ws)) return MOE_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int sms = 0;
  DeviceRestore restore;
  st = prepare_device(s, &sms, &restore);
  if (st != MOE_OK) return st;
  uint32_t* status = ws ? views_of(*shape, ws).status : nullptr;
  return cuda_status(launch_combine(*shape, Y, scatter_idx, topk_w, out, status, sms, s));
}

moe_status moe_forward(const moe_shape* shape, const float* logits, const moe_bf16* X, const moe_bf16* W_gate,
                       const moe_bf16* W_up, const moe_bf16* W_down, moe_bf16* out, void* ws, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {logits, X, W_gate, W_up, W_down, out, ws};
  for (const void* p : ptrs) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int sms = 0;
  DeviceRestore restore;
  st = prepare_device(s, &sms, &restore);
  if (st != MOE_OK) return st;
  const moe_shape& sh = *shape;
  const Views w = views_of(sh, ws);
  const moe_views& v = w.v;
  // routing, then the permutation and the row gather in one kernel
  if (launch_route_gather(sh, logits, X, v.topk_ids, v.topk_w, v.counts, v.off_pad, v.block_expert, v.num_blocks,
                          v.gather_idx, v.scatter_idx, w.local_rank, w.chunk_counts, w.xp,
                          ws_route_counter(w.status), w.win_done, forward_counters_of(sh), w.status, sms,
                          s) != cudaSuccess)
    return MOE_ERR_CUDA;
  // the down GEMM starts on each token window as soon as its h rows are in
  st = run_up_rows(sh, w.xp, v.counts, v.off_pad, W_gate, W_up, v.h, w, w.win_done, sms, s);
  if (st != MOE_OK) return st;
  st = run_down(sh, v.h, v.counts, v.off_pad, W_down, v.Y, w, w.win_done, sms, s);
  if (st != MOE_OK) return st;
  return cuda_status(launch_combine(sh, v.Y, v.scatter_idx, v.topk_w, out, w.status, sms, s));
}

}  // extern "C"
