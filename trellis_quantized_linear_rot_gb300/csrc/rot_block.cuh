// The input rotation of one 128-element block of one row, by one warp
// ("hip exl3: the input rotation and trellis linear for decode rows",
// section "What this changes", first bullet, and the rot_in test under
// "Checks on this head": fp32 product with suh, fp32 butterflies, a multiply
// by the fp32 scale, one rounding to fp16).
//
// Lane l holds elements 4l .. 4l+3. Butterfly stages h = 1, 2 pair elements
// inside a lane; stages h = 4 .. 64 pair lane l with lane l ^ (h / 4) through
// shuffles. Products and sums use explicitly rounded intrinsics, so nothing
// is contracted into an fma. Both the rot_in kernel and the fused rotation in
// the linear call this function, so their xr are the same bits.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tfx {

constexpr float kRotScale = 0x1.6a09e6p-4f;  // fp32 round-to-nearest of 1/sqrt(128)

// Four consecutive elements of x (fp16, fp32 or bf16 by DT = 0, 1, 2) as fp32.
template <int DT>
__device__ __forceinline__ void rot_load4(const void* x, size_t idx, float (&v)[4]) {
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

__device__ __forceinline__ float rot_bfly(float self, float partner, bool upper) {
  // lower <- a + b, upper <- a - b, where a is the lower element.
  return upper ? __fsub_rn(partner, self) : __fadd_rn(self, partner);
}

// Rotates block b (elements 128 b .. 128 b + 127) of row r of x into xr.
// Called by all 32 lanes of a warp together.
template <int DT>
__device__ __forceinline__ void rot_block_warp(const void* __restrict__ x, const __half* __restrict__ suh,
                                               __half* __restrict__ xr, int r, int b, int in_features,
                                               int lane) {
  const int col = b * 128 + lane * 4;
  const size_t idx = static_cast<size_t>(r) * in_features + col;
  float v[4];
  rot_load4<DT>(x, idx, v);
  const uint2 sraw = *reinterpret_cast<const uint2*>(suh + col);
  const __half2 s01 = *reinterpret_cast<const __half2*>(&sraw.x);
  const __half2 s23 = *reinterpret_cast<const __half2*>(&sraw.y);
  v[0] = __fmul_rn(v[0], __low2float(s01));
  v[1] = __fmul_rn(v[1], __high2float(s01));
  v[2] = __fmul_rn(v[2], __low2float(s23));
  v[3] = __fmul_rn(v[3], __high2float(s23));
  // h = 1: (0,1), (2,3); h = 2: (0,2), (1,3)
  const float t0 = __fadd_rn(v[0], v[1]), t1 = __fsub_rn(v[0], v[1]);
  const float t2 = __fadd_rn(v[2], v[3]), t3 = __fsub_rn(v[2], v[3]);
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
      v[e] = rot_bfly(v[e], p, upper);
    }
  }
  const __half2 o01 = __floats2half2_rn(__fmul_rn(v[0], kRotScale), __fmul_rn(v[1], kRotScale));
  const __half2 o23 = __floats2half2_rn(__fmul_rn(v[2], kRotScale), __fmul_rn(v[3], kRotScale));
  uint2 out;
  out.x = *reinterpret_cast<const uint32_t*>(&o01);
  out.y = *reinterpret_cast<const uint32_t*>(&o23);
  *reinterpret_cast<uint2*>(xr + idx) = out;
}

// Units [lo, hi) of the (row, block) units of a pass (unit u = row u / blocks
// per row, block u % blocks per row), taken by `nwarps` warps in turn.
template <int DT>
__device__ __forceinline__ void rot_units(const void* __restrict__ x, const __half* __restrict__ suh,
                                          __half* __restrict__ xr, long long lo, long long hi, int in_features,
                                          int warp, int nwarps, int lane) {
  const int blocks_per_row = in_features >> 7;
  for (long long u = lo + warp; u < hi; u += nwarps)
    rot_block_warp<DT>(x, suh, xr, static_cast<int>(u / blocks_per_row), static_cast<int>(u % blocks_per_row),
                       in_features, lane);
}

}  // namespace tfx
