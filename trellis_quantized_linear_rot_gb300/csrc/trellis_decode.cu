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

// Tiles -> strips: one 16-byte chunk of the strips order per thread.
// Strips order: block b of 128 outputs, then group c of four k-tiles, then
// [n-tile % 8][position][k-tile % 4]; chunk (b, c, nn, position) holds word
// w = strips_quad_word(bits, position) of the tiles (4c + kk, 8b + nn),
// kk = 0..3. The four words come from four k-tile rows of the tiles order;
// consecutive threads read words of one tile a few words apart, so the loads
// stay within a few sectors.
__global__ void __launch_bounds__(256) tiles_to_strips_kernel(const uint32_t* __restrict__ tiles,
                                                              uint4* __restrict__ strips,
                                                              long long chunks, int bits,
                                                              int groups_per_block, int n_tiles) {
  const int tile_words = 8 * bits;
  const long long row_words = static_cast<long long>(n_tiles) * tile_words;  // one k-tile row
  for (long long q = blockIdx.x * 256LL + threadIdx.x; q < chunks; q += static_cast<long long>(gridDim.x) * 256) {
    const long long tq = q / tile_words;  // (b, c, nn)
    const int w = strips_quad_word(bits, static_cast<int>(q - tq * tile_words));
    const int nn = static_cast<int>(tq & 7);
    const long long bc = tq >> 3;         // b * groups_per_block + c
    const long long b = bc / groups_per_block;
    const long long c = bc - b * groups_per_block;
    const uint32_t* src = tiles + (4 * c * n_tiles + 8 * b + nn) * tile_words + w;
    uint4 v;
    v.x = src[0];
    v.y = src[row_words];
    v.z = src[2 * row_words];
    v.w = src[3 * row_words];
    strips[q] = v;
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

cudaError_t launch_tiles_to_strips(const uint32_t* tiles, uint32_t* strips, int in_features,
                                   int out_features, int bits, cudaStream_t stream) {
  const int tile_words = 8 * bits;
  // One chunk per (block, group of four k-tiles, tile, word).
  const long long chunks = static_cast<long long>(in_features / 64) * (out_features / 16) * tile_words;
  long long grid = (chunks + 255) / 256;
  if (grid > 152LL * 16) grid = 152LL * 16;
  tiles_to_strips_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      tiles, reinterpret_cast<uint4*>(strips), chunks, bits, in_features / 64, out_features / 16);
  return cudaGetLastError();
}

cudaError_t launch_trellis_decode(const uint32_t* trellis, __half* w, int in_features,
                                  int out_features, int bits, cudaStream_t stream) {
  return dispatch_bits<DecodeLauncher>(bits, trellis, w, in_features, out_features, stream);
}

}  // namespace tfx
