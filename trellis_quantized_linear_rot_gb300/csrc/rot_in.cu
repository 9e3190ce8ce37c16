// rot_in: x * suh rotated by 128 and rounded to fp16 once ("hip exl3: the
// input rotation and trellis linear for decode rows", section "What this
// changes", first bullet). One warp rotates one 128-element block of one row
// (rot_block_warp).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "rot_block.cuh"

namespace tfx {

namespace {

template <int DT>
__global__ void __launch_bounds__(256) rot_in_kernel(const void* __restrict__ x,
                                                     const __half* __restrict__ suh,
                                                     __half* __restrict__ xr, int rows,
                                                     int in_features) {
  // The linear that follows may start its prologue (its weight copies need
  // nothing from this kernel); it waits for xr before reading it.
  pdl_launch_dependents();
  // This kernel itself may have started before the kernel before it (a
  // linear still reading an xr this call overwrites, or whatever wrote x)
  // has finished: wait for it before touching memory.
  pdl_wait_prerequisites();
  const int warps_per_cta = blockDim.x >> 5;
  const long long units = static_cast<long long>(rows) * (in_features >> 7);
  rot_units<DT>(x, suh, xr, 0, units, in_features,
                static_cast<int>(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5), gridDim.x * warps_per_cta,
                threadIdx.x & 31);
}

}  // namespace

cudaError_t launch_rot_in(const void* x, int x_dtype, const __half* suh, __half* xr, int rows,
                          int in_features, int num_sms, cudaStream_t stream) {
  const long long units = static_cast<long long>(rows) * (in_features / 128);
  const int warps = 8;
  long long ctas = (units + warps - 1) / warps;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  // Programmatic stream serialisation: the launch may be processed while
  // the kernel before it finishes; the kernel waits for it before touching
  // memory.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (x_dtype) {
    case 0: return cudaLaunchKernelEx(&cfg, rot_in_kernel<0>, x, suh, xr, rows, in_features);
    case 1: return cudaLaunchKernelEx(&cfg, rot_in_kernel<1>, x, suh, xr, rows, in_features);
    default: return cudaLaunchKernelEx(&cfg, rot_in_kernel<2>, x, suh, xr, rows, in_features);
  }
}

}  // namespace tfx
