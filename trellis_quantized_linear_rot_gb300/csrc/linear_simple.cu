// The trellis linear, straightforward form: one CTA per block of 128 outputs,
// one k-tile (16 inputs) per step, no pipelining. It exists as the plain
// tcgen05 formulation of the method (decode into Tensor Memory, one MMA per
// k-tile, fp32 accumulation in Tensor Memory) and as the decode-only kernel.
//
// Method: "hip exl3: the input rotation and trellis linear for decode rows",
// section "What this changes" (second bullet): a thread decodes its tile
// values with one fp16 fma each; a row's K sums are fp32 chains in a fixed
// order; the output rotation and svh finish the block.
//
// Roles of the 128 threads: thread n owns output n of the block. Per k-tile it
// decodes W[16kt .. 16kt+15][n] and writes them to TMEM lane n (the MMA's A
// operand, M = 128 outputs, K = 16), the CTA stages the 16 x 16 slice of xr
// (rows padded to 16 with zeros) in shared memory as the B operand, and one
// thread issues tcgen05.mma (N = 16) accumulating into TMEM. Every row goes
// through the same instructions whatever the row count, so a row's bits do
// not depend on the rows beside it.
#include <cstdint>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace tfx {

namespace {

constexpr uint32_t kIdescM128N16 = idesc_f16_f32(128, 16);

// B operand (16 rows x 16 k, fp16, K-major, no swizzle): core matrix
// (k / 8, r / 8) at byte (k / 8) * 256 + (r / 8) * 128; row r % 8 at
// +16 * (r % 8); element k % 8 at +2 * (k % 8).
__device__ __forceinline__ uint32_t btile_offset(int r, int k) {
  return (k >> 3) * 256 + (r >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

template <int BITS>
__global__ void __launch_bounds__(128, 1) trellis_linear_simple_kernel(LinearPass p, int* err_flag) {
  __shared__ __align__(1024) uint8_t btile[512];
  __shared__ __align__(8) uint64_t mbar;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ float xch[16][128];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int blk = blockIdx.x;
  const int KT = p.in_features / 16;
  const int NT = p.out_features / 16;
  const uint32_t bar = smem_u32(&mbar);

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_holder), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t a_tmem = tmem;       // columns 0..7: A, 128 lanes x 16 fp16
  const uint32_t d_tmem = tmem + 16;  // columns 16..31: D, 128 lanes x 16 fp32
  const uint64_t bdesc = smem_desc_noswizzle(smem_u32(btile), 256, 128);

  const int n = tid;
  const int tile_n = blk * 8 + (n >> 4);
  const int col = n & 15;
  const int br = tid >> 3;
  const int bk = (tid & 7) * 2;

  for (int kt = 0; kt < KT; ++kt) {
    const uint32_t* tw = p.trellis + (static_cast<size_t>(kt) * NT + tile_n) * (8 * BITS);
    uint32_t a[8];
    decode_col16<BITS>([&](int w) { return __ldg(tw + w); }, col, a);
    uint32_t bv = 0;
    if (br < p.rows)
      bv = __ldg(reinterpret_cast<const uint32_t*>(p.xr + static_cast<size_t>(br) * p.in_features +
                                                   kt * 16 + bk));
    if (kt > 0) mbar_wait(bar, (kt - 1) & 1, &abort_flag);  // previous MMA has read A and B
    *reinterpret_cast<uint32_t*>(btile + btile_offset(br, bk)) = bv;
    tmem_st8(a_tmem + lane_off, a);
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (abort_flag) break;
    if (tid == 0) {
      tc_fence_after();
      mma_f16_tmemA(d_tmem, a_tmem, bdesc, kIdescM128N16, kt > 0 ? 1u : 0u);
      mma_commit(bar);
    }
  }
  if (!abort_flag) mbar_wait(bar, (KT - 1) & 1, &abort_flag);
  __syncthreads();
  if (abort_flag) {
    if (tid == 0) atomicOr(err_flag, 1);
  } else {
    tc_fence_after();
    float v[16];
    tmem_ld16(d_tmem + lane_off, v);
    block_epilogue(v, p, blk, n, xch);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 32);
}

template <int BITS>
__global__ void __launch_bounds__(128) trellis_decode_kernel(const uint32_t* __restrict__ trellis,
                                                             __half* __restrict__ w,
                                                             int out_features) {
  const int n = threadIdx.x;
  const int blk = blockIdx.x;
  const int kt = blockIdx.y;
  const int NT = out_features / 16;
  const uint32_t* tw =
      trellis + (static_cast<size_t>(kt) * NT + blk * 8 + (n >> 4)) * (8 * BITS);
  uint32_t a[8];
  decode_col16<BITS>([&](int i) { return __ldg(tw + i); }, n & 15, a);
  __half* dst = w + static_cast<size_t>(kt) * 16 * out_features + blk * 128 + n;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const __half2 h = *reinterpret_cast<const __half2*>(&a[c]);
    dst[static_cast<size_t>(2 * c) * out_features] = __low2half(h);
    dst[static_cast<size_t>(2 * c + 1) * out_features] = __high2half(h);
  }
}

template <template <int> class F, typename... Args>
cudaError_t dispatch_bits(int bits, Args&&... args) {
  switch (bits) {
    case 2: return F<2>::run(args...);
    case 3: return F<3>::run(args...);
    case 4: return F<4>::run(args...);
    case 5: return F<5>::run(args...);
    case 6: return F<6>::run(args...);
    case 8: return F<8>::run(args...);
    default: return cudaErrorInvalidValue;
  }
}

template <int BITS>
struct SimpleLauncher {
  static cudaError_t run(const LinearPass& p, int* err_flag, cudaStream_t stream) {
    trellis_linear_simple_kernel<BITS><<<p.out_features / 128, 128, 0, stream>>>(p, err_flag);
    return cudaGetLastError();
  }
};

template <int BITS>
struct DecodeLauncher {
  static cudaError_t run(const uint32_t* trellis, __half* w, int in_features, int out_features,
                         cudaStream_t stream) {
    const dim3 grid(out_features / 128, in_features / 16);
    trellis_decode_kernel<BITS><<<grid, 128, 0, stream>>>(trellis, w, out_features);
    return cudaGetLastError();
  }
};

}  // namespace

cudaError_t launch_trellis_linear_simple(const LinearPass& p, int* err_flag, cudaStream_t stream) {
  return dispatch_bits<SimpleLauncher>(p.bits, p, err_flag, stream);
}

cudaError_t launch_trellis_decode(const uint32_t* trellis, __half* w, int in_features,
                                  int out_features, int bits, cudaStream_t stream) {
  return dispatch_bits<DecodeLauncher>(bits, trellis, w, in_features, out_features, stream);
}

}  // namespace tfx
