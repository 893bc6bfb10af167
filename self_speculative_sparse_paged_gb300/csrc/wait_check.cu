// Failure-detection check: a bounded wait that runs out.
//
// Every wait of the library's kernels on an mbarrier (a TMA tile landing, an
// MMA completing, a peer CTA's state) is bounded by %globaltimer: when the
// limit passes, the kernel records VEGAS_ERR_DEVICE_TIMEOUT in the device
// error word, drains what it has in flight and returns, so a lost arrival
// never hangs the GPU.  This kernel exercises that protocol on purpose and
// safely: one thread initialises an mbarrier that nothing ever arrives on,
// with no asynchronous copy or MMA outstanding, waits on it with the given
// limit, records the timeout and returns.
#include "kernels.h"
#include "vegas_common.cuh"

namespace vegas {

__global__ void __launch_bounds__(32) bounded_wait_check_kernel(unsigned long long limit_ns,
                                                                int* err, int* outcome) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  const bool arrived = mbar_wait_for(b, 0, limit_ns);   // nobody arrives: runs out
  if (!arrived) set_error(err, kErrDeviceTimeout);
  if (outcome) *outcome = arrived ? 1 : 0;
}

cudaError_t launch_bounded_wait_check(unsigned long long limit_ns, int* err, int* outcome,
                                      cudaStream_t stream) {
  bounded_wait_check_kernel<<<1, 32, 0, stream>>>(limit_ns, err, outcome);
  return cudaGetLastError();
}

}  // namespace vegas
