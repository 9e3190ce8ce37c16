// tf_trellis_decode: the dense fp16 weights W[in][out] that the trellis
// linear decodes internally ("hip exl3: the input rotation and trellis linear
// for decode rows", "Checks on this head": the linear decodes every width's
// weights bit for bit). One CTA per (128-output block, k-tile); thread n
// decodes output n's 16 weights of that k-tile with the same device code the
// linear uses, and the warp's stores of one input row are contiguous.
#include <cstdint>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "kernels.h"

namespace tfx {

namespace {

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
  decode_col16_ptr<BITS>(tw, n & 15, a);
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
struct DecodeLauncher {
  static cudaError_t run(const uint32_t* trellis, __half* w, int in_features, int out_features,
                         cudaStream_t stream) {
    const dim3 grid(out_features / 128, in_features / 16);
    trellis_decode_kernel<BITS><<<grid, 128, 0, stream>>>(trellis, w, out_features);
    return cudaGetLastError();
  }
};

}  // namespace

cudaError_t launch_trellis_decode(const uint32_t* trellis, __half* w, int in_features,
                                  int out_features, int bits, cudaStream_t stream) {
  return dispatch_bits<DecodeLauncher>(bits, trellis, w, in_features, out_features, stream);
}

}  // namespace tfx
