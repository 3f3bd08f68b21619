// moe_check.cu -- a diagnostic kernel for the bounded waits.
//
// Every pipeline of the library waits on mbarriers through mbar_wait, which
// gives up after kWaitLimitNs, records kStatusTimeout in the workspace status
// word and returns instead of hanging.  This kernel makes that wait run out on
// purpose: one thread waits on an mbarrier that nothing arrives on.  The GPU is
// never faulted; the kernel returns after the limit and the context stays
// usable, which a caller can check by reading the status word and launching
// the layer again.
#include <cstdint>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(uint32_t* status) {
  __shared__ uint64_t never_arrived;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&never_arrived, 1);
  abort_flag = 0;
  fence_mbarrier_init();
  // Phase 0 completes only after one arrival, and none comes.
  mbar_wait(&never_arrived, 0u, &abort_flag, status);
}

}  // namespace

cudaError_t launch_wait_timeout(uint32_t* status, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

}  // namespace moe
