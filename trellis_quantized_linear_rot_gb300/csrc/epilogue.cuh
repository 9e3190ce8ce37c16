// Output epilogue of the trellis linear ("hip exl3: the input rotation and
// trellis linear for decode rows", section "What this changes": the waves'
// sums, the output rotation and svh follow CUDA's finish; "Kernel contract":
// butterflies first, then the scale): for each row, the 128 fp32 K sums of a
// block go through the seven butterfly stages h = 1..64 (lower <- a + b,
// upper <- a - b), then are multiplied by fp32 1/sqrt(128), then by fp32 svh,
// and stored as fp32 or rounded once to fp16 or bf16 (nearest, ties to even;
// the page's linear registers a 4-bit bf16-output variant beside the fp32 one).
//
// Thread n (0..127) of a 128-thread group holds output n of the block for the
// 16 row slots; stages h = 1..16 are lane shuffles, h = 32 and 64 go through
// shared memory. Only the first `rows` slots are stored; the rotation runs on
// 1, 4, 8 or 16 slots, the next count up from `rows`.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"

namespace tfx {

constexpr float kOutRotScale = 0x1.6a09e6p-4f;  // fp32 round-to-nearest of 1/sqrt(128)

__device__ __forceinline__ float butterfly(float self, float partner, bool upper) {
  return upper ? __fsub_rn(partner, self) : __fadd_rn(self, partner);
}

// `bar_id`/`nthreads` name the named barrier the 128 threads share (id 0 with
// 128 threads when they are the whole CTA).
__device__ __forceinline__ void group_sync(int bar_id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
}

// The rotation of the first R row slots, as straight-line code (no per-row
// predicates, so the shuffles of different rows overlap).
template <int R>
__device__ __forceinline__ void fwht_rows(float (&v)[16], int n, float (*xch)[128], int bar_id, int nthreads) {
  const int lane = n & 31;
#pragma unroll
  for (int m = 1; m <= 16; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float q = __shfl_xor_sync(0xffffffffu, v[r], m);
      v[r] = butterfly(v[r], q, upper);
    }
  }
#pragma unroll
  for (int m = 32; m <= 64; m <<= 1) {
#pragma unroll
    for (int r = 0; r < R; ++r) xch[r][n] = v[r];
    group_sync(bar_id, nthreads);
    const bool upper = (n & m) != 0;
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = butterfly(v[r], xch[r][n ^ m], upper);
    group_sync(bar_id, nthreads);
  }
}

// The rotation of the first `rows` (1..16) row slots. It runs on 1, 4, 8 or
// 16 slots (the next count up); rows are independent, so the extra slots
// change nothing in the ones that are stored.
__device__ __forceinline__ void fwht_outputs(float (&v)[16], int rows, int n, float (*xch)[128],
                                             int bar_id = 0, int nthreads = 128) {
  if (rows > 8)
    fwht_rows<16>(v, n, xch, bar_id, nthreads);
  else if (rows > 4)
    fwht_rows<8>(v, n, xch, bar_id, nthreads);
  else if (rows > 1)
    fwht_rows<4>(v, n, xch, bar_id, nthreads);
  else
    fwht_rows<1>(v, n, xch, bar_id, nthreads);
}

// Stores rows row0 .. row0 + 15 of the pass (those below p.rows).
__device__ __forceinline__ void store_outputs(const float (&v)[16], const LinearPass& p, int blk,
                                              int n, int row0) {
  const int o = blk * 128 + n;
  const float sv = __half2float(p.svh[o]);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    if (row0 + r < p.rows) {
      const float t = __fmul_rn(__fmul_rn(v[r], kOutRotScale), sv);
      const size_t idx = static_cast<size_t>(row0 + r) * p.out_features + o;
      if (p.out_dtype == TF_F32)
        static_cast<float*>(p.y)[idx] = t;
      else if (p.out_dtype == TF_BF16)
        static_cast<__nv_bfloat16*>(p.y)[idx] = __float2bfloat16_rn(t);
      else
        static_cast<__half*>(p.y)[idx] = __float2half_rn(t);
    }
  }
}

__device__ __forceinline__ void block_epilogue(float (&v)[16], const LinearPass& p, int blk, int n,
                                               float (*xch)[128], int bar_id = 0,
                                               int nthreads = 128, int row0 = 0) {
  fwht_outputs(v, p.rows - row0 < 16 ? p.rows - row0 : 16, n, xch, bar_id, nthreads);
  store_outputs(v, p, blk, n, row0);
}

// A pass of SLOTS row slots (16 or 32): the rotation and stores run 16 row
// slots at a time, each row on its own.
template <int SLOTS>
__device__ __forceinline__ void block_epilogue_slots(float (&v)[SLOTS], const LinearPass& p, int blk, int n,
                                                     float (*xch)[128], int bar_id, int nthreads) {
#pragma unroll
  for (int h = 0; h < SLOTS; h += 16) {
    if (h < p.rows)
      block_epilogue(*reinterpret_cast<float(*)[16]>(&v[h]), p, blk, n, xch, bar_id, nthreads, h);
  }
}

}  // namespace tfx
