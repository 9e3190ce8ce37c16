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

// Generic width: the thread's words w[0..kWords) start at word
// row_first_bit(n) / 32 (circularly); they are first aligned so that the
// first window starts at the top bit, then window j is cut out at bit j*bits.
template <int BITS>
__device__ __forceinline__ void decode_words_generic(const uint32_t (&wv)[RowSpan<BITS>::kWords], int n,
                                                     uint32_t (&out)[8]) {
  using S = RowSpan<BITS>;
  const int off = row_first_bit<BITS>(n) & 31;
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

// 4 bits: a tile is 32 words; output column n's windows start at stream bit
// 64n - 12, i.e. at bit 20 of word a = (2n - 1) mod 32, and run through words
// b = 2n and c = 2n + 1; window j covers bits [20 + 4j, 36 + 4j) of a:b:c.
// Each window is cut out with one byte permute, shift or mask from a word
// or a funnel-shifted pair, six helper shifts serving all sixteen.
__device__ __forceinline__ uint32_t lo16(uint32_t x) { return x & 0xFFFFu; }
__device__ __forceinline__ uint32_t hi16(uint32_t x) { return x >> 16; }
__device__ __forceinline__ uint32_t mid16(uint32_t x) { return __byte_perm(x, 0u, 0x4421); }

__device__ __forceinline__ void decode_col16_b4(uint32_t a, uint32_t b, uint32_t c, uint32_t (&out)[8]) {
  const uint32_t p = __funnelshift_l(b, a, 12);   // stream bits 12..43 (of a:b:c)
  const uint32_t m = __funnelshift_l(b, a, 16);   // 16..47
  const uint32_t b4 = b >> 4;                     // 28..59, top nibble zero
  const uint32_t p2 = __funnelshift_l(c, b, 12);  // 44..75
  const uint32_t m2 = __funnelshift_l(c, b, 16);  // 48..79
  const uint32_t c4 = c >> 4;                     // 60..91
  const uint32_t st[16] = {mid16(p),  mid16(m),  lo16(p),  hi16(b), mid16(b4), mid16(b),
                           lo16(b4),  lo16(b),   mid16(p2), mid16(m2), lo16(p2), hi16(c),
                           mid16(c4), mid16(c),  lo16(c4), lo16(c)};
  uint32_t h[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) h[j] = mul1_half_plus_1024(st[j]);
#pragma unroll
  for (int k = 0; k < 8; ++k) out[k] = mul1_pair(h[2 * k], h[2 * k + 1]);
}

// 2 bits: a tile is 16 words; output column n's windows start at stream bit
// 32n - 14, i.e. at bit 18 of word a = (n - 1) mod 16, and run through word
// b = n; window j covers bits [18 + 2j, 34 + 2j) of a:b. The windows fall
// into four classes by their start modulo 8 bits; each class is cut out of
// one or two helper words that align it on a byte, seven helpers serving
// all sixteen (the generic cut takes two shifts per window).
__device__ __forceinline__ void decode_col16_b2(uint32_t a, uint32_t b, uint32_t (&out)[8]) {
  const uint32_t x2 = __funnelshift_l(b, a, 18);  // stream bits 18..49 (of a:b)
  const uint32_t x4 = __funnelshift_l(b, a, 20);  // 20..51
  const uint32_t x6 = __funnelshift_l(b, a, 22);  // 22..53
  const uint32_t m = __funnelshift_l(b, a, 16);   // 16..47
  const uint32_t y2 = b << 2;                     // 34..63, then zeros
  const uint32_t y4 = b << 4;                     // 36..63
  const uint32_t y6 = b << 6;                     // 38..63
  const uint32_t st[16] = {hi16(x2),  hi16(x4),  hi16(x6),  mid16(m),  mid16(x2), mid16(x4), mid16(x6), hi16(b),
                           lo16(x2),  lo16(x4),  lo16(x6),  mid16(b),  mid16(y2), mid16(y4), mid16(y6), lo16(b)};
  uint32_t h[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) h[j] = mul1_half_plus_1024(st[j]);
#pragma unroll
  for (int k = 0; k < 8; ++k) out[k] = mul1_pair(h[2 * k], h[2 * k + 1]);
}

// The 16-bit window that starts at bit P (0..31, counted from the top) of
// word `hi` and runs on into word `lo` when P > 16: one instruction where it
// sits on a byte boundary inside `hi`, two otherwise.
template <int P>
__device__ __forceinline__ uint32_t window16(uint32_t hi, uint32_t lo) {
  static_assert(P >= 0 && P < 32, "window start");
  if constexpr (P == 0) return hi16(hi);
  else if constexpr (P == 8) return mid16(hi);
  else if constexpr (P == 16) return lo16(hi);
  else if constexpr (P < 16) return (hi >> (16 - P)) & 0xFFFFu;
  else if constexpr (P == 24) return mid16(__funnelshift_l(lo, hi, 16));
  else return __funnelshift_l(lo, hi, P) >> 16;
}

// 6 bits: a tile is 48 words; output column n's windows start at stream bit
// 96n - 10, i.e. at bit 22 of word a = (3n - 1) mod 48, and run through
// words b, c, d = 3n .. 3n+2; window j covers bits [22 + 6j, 38 + 6j) of
// a:b:c:d. Windows 3, 7 and 15 sit on byte boundaries inside a word (one
// instruction each), the others take two.
template <int J>
__device__ __forceinline__ uint32_t window_b6(const uint32_t (&w)[4]) {
  constexpr int kStart = 22 + 6 * J;
  constexpr int kWord = kStart / 32;
  return window16<kStart % 32>(w[kWord], w[kWord < 3 ? kWord + 1 : 3]);
}

__device__ __forceinline__ void decode_col16_b6(const uint32_t (&w)[4], uint32_t (&out)[8]) {
  const uint32_t st[16] = {window_b6<0>(w),  window_b6<1>(w),  window_b6<2>(w),  window_b6<3>(w),
                           window_b6<4>(w),  window_b6<5>(w),  window_b6<6>(w),  window_b6<7>(w),
                           window_b6<8>(w),  window_b6<9>(w),  window_b6<10>(w), window_b6<11>(w),
                           window_b6<12>(w), window_b6<13>(w), window_b6<14>(w), window_b6<15>(w)};
  uint32_t h[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) h[j] = mul1_half_plus_1024(st[j]);
#pragma unroll
  for (int k = 0; k < 8; ++k) out[k] = mul1_pair(h[2 * k], h[2 * k + 1]);
}

// 8 bits: a tile is 64 words; output column n's windows start at stream bit
// 128n - 8, i.e. at bit 24 of word a = (4n - 1) mod 64, and run through words
// b..e = 4n .. 4n+3; window j covers bits [24 + 8j, 40 + 8j) of a:b:c:d:e, so
// every window is byte aligned: one byte permute, shift or mask each, plus a
// funnel shift for each of the four windows that straddle two words.
__device__ __forceinline__ void decode_col16_b8(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                                uint32_t e, uint32_t (&out)[8]) {
  const uint32_t ab = __funnelshift_l(b, a, 16);
  const uint32_t bc = __funnelshift_l(c, b, 16);
  const uint32_t cd = __funnelshift_l(d, c, 16);
  const uint32_t de = __funnelshift_l(e, d, 16);
  const uint32_t st[16] = {mid16(ab), hi16(b), mid16(b), lo16(b), mid16(bc), hi16(c), mid16(c), lo16(c),
                           mid16(cd), hi16(d), mid16(d), lo16(d), mid16(de), hi16(e), mid16(e), lo16(e)};
  uint32_t h[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) h[j] = mul1_half_plus_1024(st[j]);
#pragma unroll
  for (int k = 0; k < 8; ++k) out[k] = mul1_pair(h[2 * k], h[2 * k + 1]);
}

// Two-step form used by the pipelined linear: first every word a column
// needs (loads only), then the arithmetic, so a thread can issue the loads of
// several k-tiles before it needs any of them.
template <int BITS>
struct ColWords {
  static constexpr int kCount =
      BITS == 2 ? 2 : (BITS == 4 ? 3 : (BITS == 6 ? 4 : (BITS == 8 ? 5 : RowSpan<BITS>::kWords)));
  uint32_t w[kCount];
};

template <int BITS>
__device__ __forceinline__ void load_col_words(const uint32_t* tw, int n, ColWords<BITS>& cw) {
  if constexpr (BITS == 2) {
    cw.w[0] = tw[(n + 15) & 15];
    cw.w[1] = tw[n];
  } else if constexpr (BITS == 4) {
    cw.w[0] = tw[(2 * n + 31) & 31];
    const uint2 bc = *reinterpret_cast<const uint2*>(tw + 2 * n);
    cw.w[1] = bc.x;
    cw.w[2] = bc.y;
  } else if constexpr (BITS == 6) {
    cw.w[0] = tw[n == 0 ? 47 : 3 * n - 1];
#pragma unroll
    for (int j = 0; j < 3; ++j) cw.w[1 + j] = tw[3 * n + j];
  } else if constexpr (BITS == 8) {
    cw.w[0] = tw[(4 * n + 63) & 63];
    const uint4 be = *reinterpret_cast<const uint4*>(tw + 4 * n);
    cw.w[1] = be.x;
    cw.w[2] = be.y;
    cw.w[3] = be.z;
    cw.w[4] = be.w;
  } else {
    using S = RowSpan<BITS>;
    const int w0 = row_first_bit<BITS>(n) >> 5;
#pragma unroll
    for (int j = 0; j < S::kWords; ++j) {
      int wi = w0 + j;
      wi = (wi >= S::kTileWords) ? wi - S::kTileWords : wi;
      cw.w[j] = tw[wi];
    }
  }
}

template <int BITS>
__device__ __forceinline__ void decode_col_words(const ColWords<BITS>& cw, int n, uint32_t (&out)[8]) {
  if constexpr (BITS == 2) {
    decode_col16_b2(cw.w[0], cw.w[1], out);
  } else if constexpr (BITS == 4) {
    decode_col16_b4(cw.w[0], cw.w[1], cw.w[2], out);
  } else if constexpr (BITS == 6) {
    decode_col16_b6(cw.w, out);
  } else if constexpr (BITS == 8) {
    decode_col16_b8(cw.w[0], cw.w[1], cw.w[2], cw.w[3], cw.w[4], out);
  } else {
    decode_words_generic<BITS>(cw.w, n, out);
  }
}

// Decodes column n of the tile at `tw` (a pointer into shared or global
// memory), using the fast path where one exists.
template <int BITS>
__device__ __forceinline__ void decode_col16_ptr(const uint32_t* tw, int n, uint32_t (&out)[8]) {
  ColWords<BITS> cw;
  load_col_words<BITS>(tw, n, cw);
  decode_col_words<BITS>(cw, n, out);
}

// ---------------------------------------------------------------------------
// Fragment form for mma.sync.m16n8k16 with A = W^T (16 outputs x 16 inputs).
// Lane (g, t) = (lane / 4, lane % 4) owns outputs g and g + 8 of the tile at
// inputs 4t .. 4t+3 (the MMA's k positions 2t, 2t+1, 2t+8, 2t+9 are mapped to
// those four inputs; the B operand uses the same map). A group of four
// consecutive stream weights of output n starts at stream bit
// (16n + 4t) * bits + bits - 16 and spans 3 * bits + 16 bits.
template <int BITS>
struct Group4 {
  static constexpr int kTileWords = 8 * BITS;
  static constexpr int kTileBits = 256 * BITS;
  static constexpr int kWords = (3 * BITS + 16 + 31 <= 64) ? 2 : 3;
};

// Where a lane's group of four stream weights starts: word index and bit
// offset inside it (per lane constants, computed once).
template <int BITS>
struct Group4Pos {
  int w0, w1, w2, off;
  __device__ __forceinline__ Group4Pos(int n, int t) {
    using G = Group4<BITS>;
    const int start = ((16 * n + 4 * t) * BITS + BITS - 16 + G::kTileBits) % G::kTileBits;
    w0 = start >> 5;
    off = start & 31;
    w1 = (w0 + 1 == G::kTileWords) ? 0 : w0 + 1;
    w2 = (w1 + 1 == G::kTileWords) ? 0 : w1 + 1;
  }
};

// The words a group needs (loads only).
template <int BITS>
struct Group4Words {
  uint32_t x[Group4<BITS>::kWords];
};

template <int BITS>
__device__ __forceinline__ void load_group4(const uint32_t* tw, const Group4Pos<BITS>& q, Group4Words<BITS>& gw) {
  gw.x[0] = tw[q.w0];
  gw.x[1] = tw[q.w1];
  if constexpr (Group4<BITS>::kWords == 3) gw.x[2] = tw[q.w2];
}

template <int KK>
__device__ __forceinline__ uint32_t quad_word(const uint4& v) {
  if constexpr (KK == 0) return v.x;
  if constexpr (KK == 1) return v.y;
  if constexpr (KK == 2) return v.z;
  return v.w;
}

// The strips order keeps, for each tile and group of four consecutive
// k-tiles, the tile's 8 * bits word quads (word w of the four k-tiles, 16
// bytes) together, in an order chosen so that the 16 threads that decode the
// tile's columns read them with 128-bit shared-memory loads free of bank
// conflicts. A thread's i-th word of a group is word (row_first_bit(n) / 32 +
// i) mod 8 bits; at 4 and 8 bits these start every s = bits / 2 words, so
// the quads are dealt out by w mod s: quad w sits at position
// (w mod s) * (8 bits / s) + w / s, which makes the threads' i-th quads
// consecutive. The other widths keep the plain order (at 2 and 6 bits the
// threads' quads already fall in distinct banks; at 3 and 5 bits two
// threads of eight share a bank).
__host__ __device__ constexpr int strips_quad_spread(int bits) { return (bits == 4 || bits == 8) ? bits / 2 : 1; }

__host__ __device__ constexpr int strips_quad_pos(int bits, int w) {
  return (w % strips_quad_spread(bits)) * (8 * bits / strips_quad_spread(bits)) + w / strips_quad_spread(bits);
}

// The word held at position `pos` (the inverse of strips_quad_pos).
__host__ __device__ constexpr int strips_quad_word(int bits, int pos) {
  return (pos % (8 * bits / strips_quad_spread(bits))) * strips_quad_spread(bits) +
         pos / (8 * bits / strips_quad_spread(bits));
}

// Column form over the strips order: the word quads column n needs for four
// consecutive k-tiles, one 128-bit load each, then k-tile KK's words out of
// them.
template <int BITS>
struct ColQuads {
  uint4 q[ColWords<BITS>::kCount];
};

template <int BITS>
__device__ __forceinline__ void load_col_quads(const uint4* tq, int n, ColQuads<BITS>& cq) {
  if constexpr (BITS == 2) {
    cq.q[0] = tq[(n + 15) & 15];  // word n - 1 (mod 16)
    cq.q[1] = tq[n];              // word n
  } else if constexpr (BITS == 4) {
    cq.q[0] = tq[16 + ((n + 15) & 15)];  // word 2n - 1 (mod 32)
    cq.q[1] = tq[n];                     // word 2n
    cq.q[2] = tq[16 + n];                // word 2n + 1
  } else if constexpr (BITS == 6) {
    cq.q[0] = tq[n == 0 ? 47 : 3 * n - 1];  // word 3n - 1 (mod 48)
#pragma unroll
    for (int j = 0; j < 3; ++j) cq.q[1 + j] = tq[3 * n + j];
  } else if constexpr (BITS == 8) {
    cq.q[0] = tq[48 + ((n + 15) & 15)];  // word 4n - 1 (mod 64)
#pragma unroll
    for (int j = 0; j < 4; ++j) cq.q[1 + j] = tq[16 * j + n];  // word 4n + j
  } else {
    using S = RowSpan<BITS>;
    const int w0 = row_first_bit<BITS>(n) >> 5;
#pragma unroll
    for (int j = 0; j < S::kWords; ++j) {
      int wi = w0 + j;
      wi = (wi >= S::kTileWords) ? wi - S::kTileWords : wi;
      cq.q[j] = tq[wi];
    }
  }
}

template <int BITS, int KK>
__device__ __forceinline__ void quads_to_col_words(const ColQuads<BITS>& cq, ColWords<BITS>& cw) {
#pragma unroll
  for (int i = 0; i < ColWords<BITS>::kCount; ++i) cw.w[i] = quad_word<KK>(cq.q[i]);
}

// The arithmetic: packs weights (4t, 4t+1) and (4t+2, 4t+3) as two half2 words.
template <int BITS>
__device__ __forceinline__ void decode_group4_words(const Group4Words<BITS>& gw, int off, uint32_t& lo,
                                                    uint32_t& hi) {
  uint32_t s[4];
  if constexpr (Group4<BITS>::kWords == 2) {
    const uint32_t p = __funnelshift_l(gw.x[1], gw.x[0], off);  // first window at the top
    if constexpr (BITS == 4) {
      const uint32_t p4 = p >> 4;
      s[0] = hi16(p);
      s[1] = mid16(p4);
      s[2] = mid16(p);
      s[3] = lo16(p4);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) s[j] = (p >> (16 - j * BITS)) & 0xFFFFu;
    }
  } else {
    const uint32_t a0 = __funnelshift_l(gw.x[1], gw.x[0], off);
    const uint32_t a1 = __funnelshift_l(gw.x[2], gw.x[1], off);
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] = __funnelshift_l(a1, a0, j * BITS) >> 16;
  }
  lo = mul1_pair(mul1_half_plus_1024(s[0]), mul1_half_plus_1024(s[1]));
  hi = mul1_pair(mul1_half_plus_1024(s[2]), mul1_half_plus_1024(s[3]));
}

}  // namespace tfx
