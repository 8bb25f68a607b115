// Diagnostic: proves on the GPU that a pipeline wait which never completes is bounded, is
// reported through fa_sync_status, and leaves the CUDA context usable.  The kernel waits on an
// mbarrier that nothing ever arrives at, with a caller-chosen limit, using the same bounded
// wait every pipeline of the library uses.  No fault, trap or hang is involved.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {

__global__ void __launch_bounds__(32, 1) selftest_wait_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);          // expects one arrival that is never made
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait_limit(&bar, 0, &abort_flag, 900, limit_ns);
  __syncwarp();
}

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream) {
  log_launch("selftest_wait_kernel", static_cast<unsigned long long>(1), 32, static_cast<unsigned long long>(0));
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

}  // namespace fa

FA_DEFINE_STATUS_FETCH(status_fetch_selftest)
