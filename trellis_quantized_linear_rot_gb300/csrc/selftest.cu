// A self-test of the kernels' failure path: one bounded shared-memory
// barrier wait that nothing completes. The wait gives up after the same
// limit the library's kernels use, records the give-up in the device error
// flag and returns, so the host sees TF_ERR_TIMEOUT from tf_device_error and
// the CUDA context stays usable. Nothing faults, traps or hangs.
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace tfx {

namespace {

__global__ void __launch_bounds__(32) stranded_wait_kernel(int* err_flag) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none ever comes
    fence_barrier_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, &abort_flag)) atomicOr(err_flag, 1);
}

}  // namespace

cudaError_t launch_stranded_wait(int* err_flag, cudaStream_t stream) {
  stranded_wait_kernel<<<1, 32, 0, stream>>>(err_flag);
  return cudaGetLastError();
}

}  // namespace tfx
