// Self-test of the bounded on-chip waits (failure detection without a fault).
//
// Every kernel of the library waits on mbarriers through kda::mbar_wait, which
// gives up after kWaitLimitNs of wall clock, raises the CTA's abort flag and
// lets the kernel report KDA_DEVERR_TIMEOUT and return.  This kernel exercises
// exactly that path: one CTA initialises an mbarrier that nothing will
// complete, every thread waits on it, the wait runs out, and thread 0 ORs
// KDA_DEVERR_TIMEOUT into the caller's error word.  No trap, no fault; the
// context stays usable.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_device.cuh"

namespace kda {
namespace selftest {

__global__ void __launch_bounds__(128) wait_timeout_kernel(int32_t *err) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none will come
    abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0u, &abort_flag);
  __syncthreads();
  if (threadIdx.x == 0 && (!ok || abort_flag)) atomicOr(err, KDA_DEVERR_TIMEOUT);
}

}  // namespace selftest
}  // namespace kda

extern "C" int kda_selftest_wait_timeout(int32_t *err, void *stream) {
  if (!err) return KDA_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(err) & 3u) return KDA_ERR_ALIGNMENT;
  kda::selftest::wait_timeout_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(err);
  return cudaGetLastError() == cudaSuccess ? KDA_SUCCESS : KDA_ERR_LAUNCH;
}
