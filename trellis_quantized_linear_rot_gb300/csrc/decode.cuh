// Trellis decode on the GPU: one thread decodes the 16 weights one output
// column n of a 16x16 tile holds (stream weights 16n .. 16n+15) and packs them
// as 8 half2 words, word c holding input rows 2c (low half) and 2c+1.
//
// Format ("hip exl3: the input rotation and trellis linear for decode rows",
// section "What this changes": 16 x 16 tiles, 2..8 bits, mul1 with one fp16
// fma per weight): a tile is a circular stream of 256*bits bits stored in
// 8*bits uint32 words, bit j being bit (31 - j % 32) of word j / 32; weight
// i's 16-bit state is the stream bits ending at bit (i+1)*bits; mul1 maps
// state -> u = state * 0x83DCD12D mod 2^32 -> s = byte sum of u -> fp16
// fma(s, 0x1EEE, 0xC2E8).
//
// The byte sum comes out of dp4a with an addend of 0x6400, so the low half of
// the result is the fp16 number 1024 + s (exact for s <= 1020); the fma then
// uses the bias 0xC931 = 0xC2E8 - 1024 * 0x1EEE (exactly -10.3828125), which
// gives the same exact value s * a + b before the fma's single rounding.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace tfx {

constexpr uint32_t kMul1Multiplier = 0x83DCD12Du;
constexpr uint16_t kMul1ScaleBits = 0x1EEE;        // 0.00676727294921875
constexpr uint16_t kMul1BiasPlus1024Bits = 0xC931; // -3.453125 - 1024 * scale

__device__ __forceinline__ uint32_t mul1_half_plus_1024(uint32_t state16) {
  const uint32_t u = state16 * kMul1Multiplier;
  return __dp4a(u, 0x01010101u, 0x6400u);  // low 16 bits: fp16(1024 + byte sum)
}

__device__ __forceinline__ uint32_t mul1_pair(uint32_t h_lo, uint32_t h_hi) {
  const uint32_t packed = __byte_perm(h_lo, h_hi, 0x5410);
  const __half2 scale = __halves2half2(__ushort_as_half(kMul1ScaleBits), __ushort_as_half(kMul1ScaleBits));
  const __half2 bias = __halves2half2(__ushort_as_half(kMul1BiasPlus1024Bits),
                                      __ushort_as_half(kMul1BiasPlus1024Bits));
  const __half2 w = __hfma2(*reinterpret_cast<const __half2*>(&packed), scale, bias);
  return *reinterpret_cast<const uint32_t*>(&w);
}

// Words a thread reads: enough to cover the first window's bit offset inside
// its first word (up to 31) plus 15 * bits + 16 bits of windows, plus one
// word of slack so every funnel shift below has a defined second operand.
template <int BITS>
struct RowSpan {
  static constexpr int kTileWords = 8 * BITS;
  static constexpr int kTileBits = 256 * BITS;
  static constexpr int kLastWord = (15 * BITS) / 32;  // word of the last window start
  static constexpr int kWords = kLastWord + 3;
};

// Bit position (0 .. 256*bits-1) where the first window of output column n
// (weight 16n) starts.
template <int BITS>
__device__ __forceinline__ int row_first_bit(int n) {
  return (16 * n * BITS + BITS - 16 + RowSpan<BITS>::kTileBits) % RowSpan<BITS>::kTileBits;
}

// Decodes output column n (0..15) of the tile whose words start at `tw`.
// `Load` reads word w (0 <= w < 8*bits) of the tile.
template <int BITS, typename Load>
__device__ __forceinline__ void decode_col16(Load load, int n, uint32_t (&out)[8]) {
  using S = RowSpan<BITS>;
  const int p0 = row_first_bit<BITS>(n);
  const int w0 = p0 >> 5;
  const int off = p0 & 31;
  uint32_t wv[S::kWords];
#pragma unroll
  for (int j = 0; j < S::kWords; ++j) {
    int wi = w0 + j;
    wi = (wi >= S::kTileWords) ? wi - S::kTileWords : wi;
    wv[j] = load(wi);
  }
  // Align so that stream bit p0 is the most significant bit of a[0].
  uint32_t a[S::kWords - 1];
#pragma unroll
  for (int j = 0; j < S::kWords - 1; ++j) a[j] = __funnelshift_l(wv[j + 1], wv[j], off);
  uint32_t h[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int q = (j * BITS) >> 5;
    const int o = (j * BITS) & 31;
    const uint32_t state = __funnelshift_l(a[q + 1], a[q], o) >> 16;
    h[j] = mul1_half_plus_1024(state);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) out[c] = mul1_pair(h[2 * c], h[2 * c + 1]);
}

}  // namespace tfx
