// Test hook for the bounded waits: a one-CTA kernel that waits, through the
// same Watchdog / mbar_wait used by every pipeline kernel, on an mbarrier no
// thread ever arrives on.  The wait gives up after the given limit, records
// CB_ERR_TIMEOUT in the device error word, raises the CTA's abort flag (the
// other threads then stop waiting too) and the kernel returns normally: the
// failure is reported without a hang, a trap or a fault, and the context
// stays usable.
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"

namespace cb {

__global__ void __launch_bounds__(64) timeout_probe_kernel(int* err, uint64_t limit_ns) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ uint64_t never;  // no thread arrives on it
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Watchdog wd{err, &abort_flag, limit_ns};
  (void)mbar_wait(&never, 0, wd);
}

cudaError_t launch_timeout_probe(int* err, uint64_t limit_ns, cudaStream_t s) {
  return launch_pdl(timeout_probe_kernel, dim3(1), dim3(64), 0, s, err, limit_ns);
}

}  // namespace cb
