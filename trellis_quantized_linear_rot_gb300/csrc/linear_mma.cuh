// The trellis linear for decode rows on GB300, the mma.sync form: a
// persistent kernel with a TMA-fed shared-memory pipeline; the weights are
// decoded straight into tensor-core operand registers and multiplied with
// mma.sync.m16n8k16. It runs the no-allocation entry point's passes of up to
// 16 rows, whose scratch has room for its 2 x 16 x 128 partial sums per CTA
// but not for the tcgen05 kernel's (linear_tc.cuh), which runs every other
// pass. Both kernels give every row the same bits.
//
// Method: "hip exl3: the input rotation and trellis linear for decode rows",
// section "What this changes" (second bullet): the trellis linear at 2..8 bits
// with mul1, one fp16 fma per decoded weight, each row's K sums in a fixed
// order (so a row's bits do not depend on the rows sharing its launch), no
// bias; the output rotation and svh finish each 128-output block.
//
// mma.sync.m16n8k16 (2.2 cycles per instruction per SM) takes the A operand
// straight from the decode registers and is issued by every compute warp, so
// the contraction spreads over all four sub-partitions; the tcgen05 kernel
// stages the decoded weights through Tensor Memory instead and is faster at
// every row count measured (LM head 4 bits: 120.5 against 137 us at 1 row).
//
// Work: the (output block b, 128-input unit) grid, block-major, is cut into
// one contiguous range per CTA (one CTA per SM). Consecutive units of one block
// form a segment; a segment's sums accumulate in registers in input order. A
// block whose units all belong to one CTA is finished by it; a block cut
// between CTAs has each CTA publish its partial sums, and the CTA that arrives
// last adds them in CTA order (the input order) and finishes the block. The
// cut depends only on the shape and the CTA count, never on the rows.
//
// Warp roles:
//   warps 0-3   epilogue: sums of a finished segment (from shared memory) ->
//               output rotation -> svh -> y, or the cross-CTA partial sums
//   warps 4-19  compute, two groups of 8: warp 4 + 8q + j of group q owns output
//               tile j (outputs 16j..16j+15 of the block); group q takes the
//               units q, q + 2, ... of each segment; per unit a warp decodes its
//               8 tiles (one per k-tile) into A fragments and issues one
//               mma.sync per 8 rows per tile; a segment's sum is group 0's
//               plus group 1's, added in that order
//   warp 20     producer: one thread issues the TMA copies of each unit
//               (packed weights of 8 k-tiles x 8 tiles; the 16 x 128 slice of
//               xr, 128-byte swizzled so the B-fragment loads hit distinct
//               banks)
// All waits are bounded; a kernel that gives up sets the error flag and exits.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "decode.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "per_device.h"
#include "ptx.cuh"

namespace tfx {

namespace {

constexpr int kTileWarps = 8;        // one per 16-output tile of a block
constexpr int kGroups = 2;           // compute groups of 8 warps, alternating units
constexpr int kComputeWarps = kTileWarps * kGroups;
constexpr int kThreads = (4 + kComputeWarps + 1) * 32;
constexpr int kSmemBudget = 196 * 1024;
constexpr int kSmemBudgetWide = 227 * 1024;  // the per-block maximum (the tcgen05 kernel)

// A pass of up to 8 * NB rows (NB = 1 or 2): its MMAs cover NB blocks of 8
// row slots; its sums and xr slices have room for 16 row slots.
template <int NB>
struct Slots {
  static_assert(NB == 1 || NB == 2, "passes of up to 16 rows");
  static constexpr int kRows = 16;
};

// A unit is UKT k-tiles (16 * UKT inputs) of one output block: 8, or 16 when
// the input count allows (fewer synchronisations per weight).
template <int BITS, int UKT, int NB>
struct Cfg {
  static constexpr int kSlots = Slots<NB>::kRows;
  static constexpr int kWUnitBytes = 256 * BITS * UKT;  // UKT k-tiles x 8 tiles x 32*BITS bytes
  static constexpr int kXrChunkBytes = 128 * kSlots;    // one 64-input chunk of the xr slice
  static constexpr int kXrUnitBytes = kXrChunkBytes * (UKT / 4);
  static constexpr int kStageBytes = kWUnitBytes + kXrUnitBytes;
  static constexpr int kDbufBytes = 2 * kGroups * kSlots * 128 * 4;  // [2][groups][slots][128] fp32
  static constexpr int kStagesFit = (kSmemBudget - kDbufBytes - 8192 - 1024) / kStageBytes;
  // Even, so that unit k and unit k - kStages (the stage's previous unit)
  // always belong to the same compute group (see the kernel).
  static constexpr int kStages = (kStagesFit < 12 ? kStagesFit : 12) & ~1;
};

struct MmaParams {
  const uint8_t* strips;  // packed weights in strips order (strips layout only)
  const __half* svh;
  void* y;
  float* partials;      // this kernel: [ctas][2][16][128]; the tcgen05 kernel: [ctas][3][128][128]
  int* counters;        // [out_features / 128]
  int* err_flag;
  long long units;      // (out/128) * (in/128)
  int units_per_block;  // in / 128
  int ctas;
  int out_dtype;  // TF_F16, TF_F32 or TF_BF16
  int rows;
  int in_features;
  int out_features;
  // The fused rotation (tcgen05 kernel only): null rot_x for none.
  const void* rot_x = nullptr;
  const __half* rot_suh = nullptr;
  __half* rot_xr = nullptr;
  int* rot_sync = nullptr;
  int rot_dtype = 0;
};

__device__ __forceinline__ long long range_start(long long c, long long units, int ctas) {
  return c * units / ctas;
}

// CTA whose range holds unit u.
__device__ __forceinline__ int cta_of_unit(long long u, long long units, int ctas) {
  return static_cast<int>(((u + 1) * ctas - 1) / units);
}

// Slot of a CTA's partial sums for block b: 0 for the first block of its
// range, 1 for the last (a CTA's range cuts at most two blocks).
__device__ __forceinline__ int partial_slot(int c, int b, const MmaParams& p) {
  const long long first_block = range_start(c, p.units, p.ctas) / p.units_per_block;
  return b == first_block ? 0 : 1;
}

// The order in which a CTA works through its segments (one per output block
// its range touches). When the range ends inside a block, that block is
// shared with the next CTA, which takes its own part of it first; this CTA
// then also takes that segment first, so both parts of every shared block
// are summed early and no cross-CTA sum is left for the end of the kernel.
// The order changes no result: a block's sum does not depend on when its
// segments run. Units are indexed from the range start; a segment's units
// are consecutive in the processing order, starting at pos().
struct SegmentOrder {
  long long u0, b_first, b_last;
  int UB, n_units, n_seg, n_last;
  bool rotated;
  __device__ SegmentOrder(long long u0_, long long u1_, int UB_) {
    u0 = u0_;
    UB = UB_;
    n_units = static_cast<int>(u1_ - u0_);
    b_first = u0_ / UB_;
    b_last = (u1_ - 1) / UB_;
    n_seg = static_cast<int>(b_last - b_first) + 1;
    n_last = n_units - lo(b_last);
    rotated = n_seg >= 2 && (u1_ % UB_) != 0;
  }
  __device__ long long block(int q) const {
    return rotated ? (q == 0 ? b_last : b_first + q - 1) : b_first + q;
  }
  __device__ int lo(long long bb) const { return bb * UB > u0 ? static_cast<int>(bb * UB - u0) : 0; }
  __device__ int hi(long long bb) const {
    const long long h = (bb + 1) * UB - u0;
    return h < n_units ? static_cast<int>(h) : n_units;
  }
  // Processing position of the first unit of segment q (whose first unit is lo).
  __device__ int pos(int q, int seg_lo) const { return rotated ? (q == 0 ? 0 : n_last + seg_lo) : seg_lo; }
};

// Walks the units of a CTA in processing order: block and unit within it.
struct UnitCursor {
  SegmentOrder o;
  int q, i, end;
  long long bb;
  __device__ explicit UnitCursor(const SegmentOrder& order) : o(order), q(0) {
    bb = o.block(0);
    i = o.lo(bb);
    end = o.hi(bb);
  }
  __device__ int ub() const { return static_cast<int>(o.u0 + i - bb * o.UB); }
  __device__ void next() {
    if (++i == end && ++q < o.n_seg) {
      bb = o.block(q);
      i = o.lo(bb);
      end = o.hi(bb);
    }
  }
};

template <int BITS, int UKT, int NB>
struct Layout {
  static constexpr int kStages = Cfg<BITS, UKT, NB>::kStages;
  static constexpr int kStageBytes = Cfg<BITS, UKT, NB>::kStageBytes;
  static constexpr int kDbufOff = kStages * kStageBytes;        // [2][groups][slots][128] fp32 sums
  static constexpr int kXchOff = kDbufOff + Cfg<BITS, UKT, NB>::kDbufBytes;  // [16][128] fp32 for the rotation
  static constexpr int kBarOff = kXchOff + 8192;
  static constexpr int kNumBars = 2 * kStages + 4;               // full, empty, dfull[2], dempty[2]
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kUsed = kMiscOff + 64;
  // At least 120 KB, so that two CTAs never share an SM.
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
};

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One k-tile of a compute warp: decode the lane's two runs of four weights
// into the A fragment, then one MMA per 8 row slots.
template <int BITS, int NB>
__device__ __forceinline__ void tile_step(const Group4Words<BITS>& wa, const Group4Words<BITS>& wb,
                                          const Group4Pos<BITS>& pos_a, const Group4Pos<BITS>& pos_b,
                                          const uint2 (&b)[NB], float (&d)[NB][4]) {
  uint32_t a[4];
  decode_group4_words<BITS>(wa, pos_a.off, a[0], a[2]);
  decode_group4_words<BITS>(wb, pos_b.off, a[1], a[3]);
#pragma unroll
  for (int q = 0; q < NB; ++q) mma_16816(d[q], a, b[q].x, b[q].y);
}

// B fragments of one k-tile: rows 8q + g of the xr chunk (1024 bytes apart).
template <int NB>
__device__ __forceinline__ void load_b(const uint8_t* x, uint2 (&b)[NB]) {
#pragma unroll
  for (int q = 0; q < NB; ++q) b[q] = *reinterpret_cast<const uint2*>(x + q * 1024);
}

// Weight layouts: k-tile major ("tiles": tile (kt, nt) at (kt*O/16 + nt)),
// landing in shared memory as [k-tile][8 tiles][words]; or block-contiguous
// with the words of four consecutive k-tiles interleaved ("strips": block b,
// then groups of four k-tiles, then [tile % 8][word quad][k-tile % 4], the
// quads in the order strips_quad_pos gives), landing as
// [k-tile / 4][8 tiles][word quads][k-tile % 4]. This kernel reads the
// tiles order (the no-allocation entry point's); the strips order is the
// tcgen05 kernel's.
enum { kLayoutTiles = 0, kLayoutStrips = 1 };

template <int BITS, int NB, int UKT>
__global__ void __launch_bounds__(kThreads, 1)
    trellis_linear_mma_kernel(const __grid_constant__ CUtensorMap wmap,
                              const __grid_constant__ CUtensorMap xmap, const MmaParams p) {
  using L = Layout<BITS, UKT, NB>;
  using C = Cfg<BITS, UKT, NB>;
  constexpr int kSlots = C::kSlots;
  constexpr int S = L::kStages;
  // Unit k (processing position) sits in stage k % S, phase k / S, and goes
  // to compute group k % 2. With S even, a stage's previous unit k - S went
  // to the same group, which therefore read it (so its phase completed)
  // before it waits for unit k: no wait can look two phases ahead, where a
  // parity test could not tell the phases apart.
  static_assert(S % kGroups == 0 && S >= 2 * kGroups, "a stage must stay with one compute group");
  extern __shared__ __align__(1024) uint8_t smem[];
  float* dbuf = reinterpret_cast<float*>(smem + L::kDbufOff);
  float(*xch)[128] = reinterpret_cast<float(*)[128]>(smem + L::kXchOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto dfull_bar = [&](int d) { return bar0 + 8u * (2 * S + d); };
  auto dempty_bar = [&](int d) { return bar0 + 8u * (2 * S + 2 + d); };

  // The warp index through a shuffle from lane 0, so that the compiler knows
  // it is the same in every lane (role values in uniform registers).
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  constexpr int kProducerWarp = 4 + kComputeWarps;
  const int c = blockIdx.x;
  const SegmentOrder order(range_start(c, p.units, p.ctas), range_start(c + 1, p.units, p.ctas),
                           p.units_per_block);
  const int n_units = order.n_units;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *last_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kTileWarps);  // the 8 warps of the group that takes the unit
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(dfull_bar(d), kComputeWarps);
      mbar_init(dempty_bar(d), 4);
    }
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
  }
  __syncthreads();
  // The kernel after this one may be scheduled now; it waits for this one
  // before touching memory this one reads or writes (as this one does for
  // the kernel before it).
  pdl_launch_dependents();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      UnitCursor cur(order);
      UnitCursor xcur(order);
      const uint64_t wpolicy = l2_evict_first();  // weights: first out of L2
      int s = 0;
      int round = 0;
      // The first stages' weight copies need nothing from the kernel before
      // this one (the rotation that writes xr); the xr copies wait for it.
      const int pre = n_units < S ? n_units : S;
      for (int i = 0; i < pre; ++i) {
        const uint32_t st = smem_u32(smem + i * L::kStageBytes);
        mbar_arrive_expect_tx(full_bar(i), L::kStageBytes);
        tma_load_2d(st, &wmap, static_cast<int>(cur.bb) * 32 * BITS, cur.ub() * UKT, full_bar(i), wpolicy);
        cur.next();
      }
      pdl_wait_prerequisites();
      for (int i = 0; i < pre; ++i) {
        tma_load_3d(smem_u32(smem + i * L::kStageBytes) + C::kWUnitBytes, &xmap, 0, 0, xcur.ub() * (UKT / 4),
                    full_bar(i));
        xcur.next();
      }
      issued = pre;
      s = pre == S ? 0 : pre;
      round = pre == S ? 1 : 0;
      for (int i = pre; i < n_units; ++i) {
        if (round > 0 && !mbar_wait_sleepy(empty_bar(s), (round - 1) & 1, abort_flag, 128)) break;
        const uint32_t st = smem_u32(smem + s * L::kStageBytes);
        mbar_arrive_expect_tx(full_bar(s), L::kStageBytes);
        tma_load_2d(st, &wmap, static_cast<int>(cur.bb) * 32 * BITS, cur.ub() * UKT, full_bar(s), wpolicy);
        tma_load_3d(st + C::kWUnitBytes, &xmap, 0, 0, cur.ub() * (UKT / 4), full_bar(s));
        issued = i + 1;
        cur.next();
        if (++s == S) {
          s = 0;
          ++round;
        }
      }
      // Let every copy this CTA started land before it can exit.
      for (int i = issued - S > 0 ? issued - S : 0; i < issued; ++i) {
        volatile int never = 0;
        mbar_wait(full_bar(i % S), (i / S) & 1, &never);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- compute
    const int cg = (warp - 4) / kTileWarps;  // group: takes units cg, cg + kGroups, ... of each segment
    const int j = (warp - 4) % kTileWarps;   // output tile of the block
    const int g = lane >> 2;                 // outputs g and g + 8 of the tile
    const int t = lane & 3;                  // inputs 4t .. 4t+3 of each k-tile
    // Byte offsets of this lane's B fragments inside a unit's xr slice, for
    // k-tiles kt % 4 = 0..3 (row g; row 8q + g is 1024 q bytes further):
    // 16-byte chunk c = 2 (kt % 4) + t / 2 of a 128-byte row sits at chunk
    // c ^ (row % 8).
    int xoff[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) xoff[q] = g * 128 + (((2 * q + (t >> 1)) ^ g) << 4) + (t & 1) * 8;
    const Group4Pos<BITS> pos_a(g, t);      // output g of the tile
    const Group4Pos<BITS> pos_b(g + 8, t);  // output g + 8
    bool stop = false;
    for (int sg = 0; sg < order.n_seg && !stop; ++sg) {
      const long long bb = order.block(sg);
      const int seg_lo = order.lo(bb);
      const int seg_hi = order.hi(bb);
      const int base = order.pos(sg, seg_lo) - seg_lo;  // processing position of unit i: base + i
      float d[NB][4];  // row slots 8q .. 8q+7
#pragma unroll
      for (int q = 0; q < NB; ++q) d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.f;
      // The group's units of the segment: processing positions k = base + i
      // with k % 2 == cg, in order.
      int i = seg_lo + (((cg - base - seg_lo) % kGroups) + kGroups) % kGroups;
      for (; i < seg_hi; i += kGroups) {
        const int k = base + i;
        const int s = k % S;
        const bool ok = mbar_wait_sleepy(full_bar(s), (k / S) & 1, abort_flag, 32);
        if (!__all_sync(0xffffffffu, ok)) {
          stop = true;
          break;
        }
        const uint8_t* st = smem + s * L::kStageBytes;
        const uint8_t* xs = st + C::kWUnitBytes;
        const uint32_t* wtile = reinterpret_cast<const uint32_t*>(st + j * 32 * BITS);
        // Software pipeline over k-tiles: the words and B fragments of tile
        // kt + 1 are loaded before tile kt is decoded.
        Group4Words<BITS> wa, wb;
        load_group4<BITS>(wtile, pos_a, wa);
        load_group4<BITS>(wtile, pos_b, wb);
        uint2 b[NB];
        load_b<NB>(xs + xoff[0], b);
#pragma unroll
        for (int kt = 0; kt < UKT; ++kt) {
          Group4Words<BITS> na, nb;
          uint2 nx[NB];
          if (kt + 1 < UKT) {
            const uint32_t* tn = wtile + (kt + 1) * 64 * BITS;
            load_group4<BITS>(tn, pos_a, na);
            load_group4<BITS>(tn, pos_b, nb);
            load_b<NB>(xs + ((kt + 1) >> 2) * C::kXrChunkBytes + xoff[(kt + 1) & 3], nx);
          }
          tile_step<BITS, NB>(wa, wb, pos_a, pos_b, b, d);
          if (kt + 1 < UKT) {
            wa = na;
            wb = nb;
#pragma unroll
            for (int q = 0; q < NB; ++q) b[q] = nx[q];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
      }
      if (stop) break;
      // This group's sums of the segment (zero if it took none of its units).
      const int dbi = sg & 1;
      bool ok2 = true;
      if (sg >= 2) ok2 = mbar_wait(dempty_bar(dbi), ((sg >> 1) - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok2)) break;
      // D fragment q: (output g, row 8q+2t), (g, 8q+2t+1), (g+8, 8q+2t), (g+8, 8q+2t+1).
      float* db = dbuf + (dbi * kGroups + cg) * kSlots * 128;
      const int o = 16 * j + g;
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const int r = 8 * q + 2 * t;
        db[r * 128 + o] = d[q][0];
        db[(r + 1) * 128 + o] = d[q][1];
        db[r * 128 + o + 8] = d[q][2];
        db[(r + 1) * 128 + o + 8] = d[q][3];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(dfull_bar(dbi));
    }
  } else {
    // ----------------------------------------------------------- epilogue
    pdl_wait_prerequisites();  // partial sums, counters and y follow the kernel before
    const int t = threadIdx.x;  // output within the block
    LinearPass lp;
    lp.svh = p.svh;
    lp.y = p.y;
    lp.out_dtype = p.out_dtype;
    lp.rows = p.rows;
    lp.in_features = p.in_features;
    lp.out_features = p.out_features;
    for (int sg = 0; sg < order.n_seg; ++sg) {
      const int b = static_cast<int>(order.block(sg));
      const int d = sg & 1;
      const bool ok = mbar_wait_sleepy(dfull_bar(d), (sg >> 1) & 1, abort_flag, 1000);
      if (!group_all(1, 128, ok)) break;  // the group's named barriers need all 128 threads
      float v[kSlots];
      const float* db = dbuf + d * kGroups * kSlots * 128;
#pragma unroll
      for (int r = 0; r < kSlots; ++r) v[r] = db[r * 128 + t];
#pragma unroll
      for (int q = 1; q < kGroups; ++q)  // the groups' sums, added in group order
#pragma unroll
        for (int r = 0; r < kSlots; ++r) v[r] = __fadd_rn(v[r], db[q * kSlots * 128 + r * 128 + t]);
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty_bar(d));
      const int c_first = cta_of_unit(static_cast<long long>(b) * order.UB, p.units, p.ctas);
      const int c_last = cta_of_unit(static_cast<long long>(b + 1) * order.UB - 1, p.units, p.ctas);
      if (c_first == c_last) {
        block_epilogue_slots<kSlots>(v, lp, b, t, xch, 1, 128);
        continue;
      }
      // Block shared with other CTAs: publish the partial sums, count arrivals.
      float* mine = p.partials + (static_cast<size_t>(c) * 2 + partial_slot(c, b, p)) * kSlots * 128;
#pragma unroll
      for (int r = 0; r < kSlots; ++r)
        if (r < p.rows) mine[r * 128 + t] = v[r];
      __threadfence();
      group_sync(1, 128);
      if (t == 0) {
        const int old = atomicAdd(p.counters + b, 1);
        *last_flag = (old == c_last - c_first) ? 1 : 0;
      }
      group_sync(1, 128);
      const bool last = *last_flag != 0;
      if (last) {
        __threadfence();
        for (int cc = c_first; cc <= c_last; ++cc) {
          const float* src =
              p.partials + (static_cast<size_t>(cc) * 2 + partial_slot(cc, b, p)) * kSlots * 128;
          // 16 row slots are loaded at once (slots past `rows` hold stale
          // values that are never used), so the loads overlap.
#pragma unroll
          for (int h = 0; h < kSlots; h += 16) {
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = __ldcg(src + (h + r) * 128 + t);
#pragma unroll
            for (int r = 0; r < 16; ++r)
              if (h + r < p.rows) v[h + r] = (cc == c_first) ? x[r] : __fadd_rn(v[h + r], x[r]);
          }
        }
        block_epilogue_slots<kSlots>(v, lp, b, t, xch, 1, 128);
        if (t == 0) p.counters[b] = 0;
      }
      group_sync(1, 128);
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err_flag, 1);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

constexpr int kMaxAttrDevices = 64;

// The dynamic shared-memory limit of a kernel, set once on each device that
// launches it (the attribute belongs to the current device).
template <typename Kernel>
cudaError_t smem_attr_once(PerDeviceOnce<kMaxAttrDevices>& once, Kernel kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return static_cast<cudaError_t>(once.run(dev, static_cast<int>(cudaErrorInvalidDevice), [&] {
    return static_cast<int>(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  }));
}

template <int BITS, int NB, int UKT>
cudaError_t set_smem_attr() {
  static PerDeviceOnce<kMaxAttrDevices> once;
  return smem_attr_once(once, trellis_linear_mma_kernel<BITS, NB, UKT>, Layout<BITS, UKT, NB>::kBytes);
}

template <int BITS, int NB, int UKT>
cudaError_t launch_one(const CUtensorMap& wmap, const CUtensorMap& xmap, const MmaParams& p, int ctas,
                       cudaStream_t stream) {
  cudaError_t e = set_smem_attr<BITS, NB, UKT>();
  if (e != cudaSuccess) return e;
  // Programmatic stream serialisation: this kernel may start while the
  // kernel before it (the input rotation) finishes; its producer waits for
  // that kernel's writes before it copies xr.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout<BITS, UKT, NB>::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, trellis_linear_mma_kernel<BITS, NB, UKT>, wmap, xmap, p);
}

// One pass of up to 16 rows on weights in the tiles order.
template <int BITS, int UKT>
cudaError_t run_mma(const LinearPass& lp, const TcWorkspace& ws, bool strips, cudaStream_t stream) {
  if (strips) return cudaErrorInvalidValue;  // the tcgen05 kernel's order
  if (lp.rot_x != nullptr) return cudaErrorInvalidValue;  // the fused rotation is the tcgen05 kernel's
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap wmap, xmap;
  {
    // Packed weights as rows of u64: one row per k-tile, O * BITS / 4 words.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(lp.out_features) * BITS / 4,
                                static_cast<cuuint64_t>(lp.in_features / 16)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lp.out_features) * BITS * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(32 * BITS), static_cast<cuuint32_t>(UKT)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint32_t*>(lp.trellis), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // xr [rows][in] fp16 viewed as (64 inputs, rows, in / 64): a box of
    // (64, 16, UKT / 4) lands as UKT / 4 chunks of 64 inputs, each of 16
    // row slots, 128 bytes per row, with the 128-byte swizzle; slots past
    // `rows` are zero.
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(lp.rows),
                                static_cast<cuuint64_t>(lp.in_features / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(lp.in_features) * 2, 128};
    const cuuint32_t box[3] = {64, 16u, static_cast<cuuint32_t>(UKT / 4)};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(lp.xr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  MmaParams p;
  p.strips = nullptr;
  p.svh = lp.svh;
  p.y = lp.y;
  p.partials = ws.partials;
  p.counters = ws.counters;
  p.err_flag = ws.err_flag;
  p.units_per_block = lp.in_features / (16 * UKT);
  p.units = static_cast<long long>(lp.out_features / 128) * p.units_per_block;
  p.ctas = ws.ctas;
  p.out_dtype = lp.out_dtype;
  p.rows = lp.rows;
  p.in_features = lp.in_features;
  p.out_features = lp.out_features;
  if (p.rows > 8) return launch_one<BITS, 2, UKT>(wmap, xmap, p, ws.ctas, stream);
  return launch_one<BITS, 1, UKT>(wmap, xmap, p, ws.ctas, stream);
}

}  // namespace
}  // namespace tfx
