// rot_in: x * suh rotated by 128 and rounded to fp16 once ("hip exl3: the
// input rotation and trellis linear for decode rows", section "What this
// changes", first bullet, and the rot_in test under "Checks on this head":
// fp32 product, fp32 butterflies, a multiply by the fp32 scale, one rounding).
//
// One warp rotates one 128-element block of one row: lane l holds elements
// 4l .. 4l+3. Butterfly stages h = 1, 2 pair elements inside a lane; stages
// h = 4 .. 64 pair lane l with lane l ^ (h / 4) through shuffles. Products and
// sums use explicitly rounded intrinsics, so nothing is contracted into an fma.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace tfx {

namespace {

constexpr float kRotScale = 0x1.6a09e6p-4f;  // fp32 round-to-nearest of 1/sqrt(128)

template <int DT>
__device__ __forceinline__ void load4(const void* x, size_t idx, float (&v)[4]) {
  if constexpr (DT == 0) {  // fp16
    const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const __half*>(x) + idx);
    const __half2 a = *reinterpret_cast<const __half2*>(&raw.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&raw.y);
    v[0] = __low2float(a);
    v[1] = __high2float(a);
    v[2] = __low2float(b);
    v[3] = __high2float(b);
  } else if constexpr (DT == 1) {  // fp32
    const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx);
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  } else {  // bf16
    const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(x) + idx);
    v[0] = __uint_as_float(raw.x << 16);
    v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    v[2] = __uint_as_float(raw.y << 16);
    v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float bfly(float self, float partner, bool upper) {
  // lower <- a + b, upper <- a - b, where a is the lower element.
  return upper ? __fsub_rn(partner, self) : __fadd_rn(self, partner);
}

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
  const int lane = threadIdx.x & 31;
  const int warps_per_cta = blockDim.x >> 5;
  const int blocks_per_row = in_features >> 7;
  const long long units = static_cast<long long>(rows) * blocks_per_row;
  for (long long u = static_cast<long long>(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5);
       u < units; u += static_cast<long long>(gridDim.x) * warps_per_cta) {
    const int r = static_cast<int>(u / blocks_per_row);
    const int b = static_cast<int>(u % blocks_per_row);
    const int col = b * 128 + lane * 4;
    const size_t idx = static_cast<size_t>(r) * in_features + col;
    float v[4];
    load4<DT>(x, idx, v);
    const uint2 sraw = *reinterpret_cast<const uint2*>(suh + col);
    const __half2 s01 = *reinterpret_cast<const __half2*>(&sraw.x);
    const __half2 s23 = *reinterpret_cast<const __half2*>(&sraw.y);
    v[0] = __fmul_rn(v[0], __low2float(s01));
    v[1] = __fmul_rn(v[1], __high2float(s01));
    v[2] = __fmul_rn(v[2], __low2float(s23));
    v[3] = __fmul_rn(v[3], __high2float(s23));
    // h = 1: (0,1), (2,3); h = 2: (0,2), (1,3)
    float t0 = __fadd_rn(v[0], v[1]), t1 = __fsub_rn(v[0], v[1]);
    float t2 = __fadd_rn(v[2], v[3]), t3 = __fsub_rn(v[2], v[3]);
    v[0] = __fadd_rn(t0, t2);
    v[2] = __fsub_rn(t0, t2);
    v[1] = __fadd_rn(t1, t3);
    v[3] = __fsub_rn(t1, t3);
#pragma unroll
    for (int m = 1; m <= 16; m <<= 1) {  // h = 4 m
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = __shfl_xor_sync(0xffffffffu, v[e], m);
        v[e] = bfly(v[e], p, upper);
      }
    }
    const __half2 o01 = __floats2half2_rn(__fmul_rn(v[0], kRotScale), __fmul_rn(v[1], kRotScale));
    const __half2 o23 = __floats2half2_rn(__fmul_rn(v[2], kRotScale), __fmul_rn(v[3], kRotScale));
    uint2 out;
    out.x = *reinterpret_cast<const uint32_t*>(&o01);
    out.y = *reinterpret_cast<const uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(xr + idx) = out;
  }
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
