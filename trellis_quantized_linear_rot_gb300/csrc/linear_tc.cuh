// The trellis linear on GB300 with tcgen05: the decoded weights go to
// Tensor Memory and tensor-core MMAs form the K sums of every pass, from one
// decode row up to 128 rows, with the same results bit for bit as the
// mma.sync kernel (linear_mma.cuh).
//
// Method: "hip exl3: the input rotation and trellis linear for decode rows",
// section "What this changes" (second bullet: the trellis linear for 1 to 16
// rows a pass, a row's sums in a fixed order that does not depend on the
// rows sharing its launch) and section "Known limits" (the prompt path,
// registered bit-equal to the decode linear). Bit-equality holds because
// every output element goes through the same sums in every pass and in both
// kernels: the same cut of the (block, unit) grid between CTAs, the same two
// chains per segment (the units at even and at odd processing positions,
// each a chain of K = 16 tensor-core steps in input order), their fp32 sum
// in that order, and the partial sums of a shared block added in CTA order.
// A tcgen05.mma (M = 128, K = 16, A in Tensor Memory) gives the same bits as
// mma.sync.m16n8k16 for the same operands and accumulator, also when the 16
// inputs of a step are presented in another order (checked on the GB300 over
// 81,920 outputs of chains of eight steps with wide exponent ranges).
//
// Per CTA (one per SM): the MMA's M is the 128 outputs of a block (Tensor
// Memory lanes), N the pass's row slots (rows rounded up to 16), K 16 inputs
// per k-tile.
//
// Warp roles:
//   warps 0-3   epilogue: per segment, the two chains' sums from Tensor
//               Memory, added, written to this CTA's partial-sum slot, then
//               (when the CTA owns the block, or arrives last) the output
//               rotation, svh and the stores
//   decode      six warpgroups (24 warps) in the 16-row-slot class at 4, 6
//               and 8 bits, five (20 warps) otherwise up to 32 row slots,
//               four (16 warps) beyond: they take half-units (8 k-tiles) in turn,
//               half-unit q going to warpgroup q mod kWG; thread n decodes
//               output n's 16 weights of each k-tile into Tensor Memory lane
//               n (the MMA's A operand), in its warpgroup's A buffer, whose
//               uses go to whichever chain each half-unit belongs to. More
//               decode warps per SM sub-partition leave fewer idle issue
//               slots while one of them waits (LM head 4 bits, strips, four
//               to five: 122.8 -> 120.8 us at 1 row; k-tile order, five to
//               six: 115.6 -> 114.6)
//   next warp   weights producer: one elected lane copies each half-unit's
//               packed weights into the stage ring as soon as the decode of
//               the stage's previous half-unit is done
//   next warp   xr producer: one elected lane copies each half-unit's xr slice
//               (one tensor copy of two chunks of 64 inputs x the pass's row
//               slots, with the 128-byte swizzle: the MMA's K-major B layout)
//               as soon as the MMAs of the stage's previous half-unit are done
//   last two    MMA, one warp per chain: each issues its chain's MMAs in
//               input order (one elected lane of the whole warp), a whole
//               unit's 16 at once where one copy brings the unit; the first
//               allocates Tensor Memory. One issuing thread retires about one
//               MMA (M = 128, N = 16, K = 16) per 65 cycles, and two issuing
//               warps twice as many (measured on the GB300), so each chain
//               has its own warp; one issuing warp for both chains was busy
//               most of the time and held the decode up.
// A half-unit's weights and its xr slice sit in two rings, each with its
// own depth and its own full and empty barriers: the weights are read by
// the decode and the xr slice by the MMAs, so each part is refilled as soon
// as its reader is done, by its own warp. A single thread issuing every copy was the
// kernel's bottleneck (measured on the GB300: a thread issuing 1-D bulk
// copies alone manages one copy per ~500 cycles whatever its size, most of it
// the thread's own chain of dependent instructions), so the two producers
// keep their loops short and work from counters, not divisions. Each runs
// its loop on the whole warp, like the MMA warps, so that the copies'
// operands are warp-uniform: the same loop on lane 0 alone issued more
// instructions, which the decode warps of its sub-partition paid for.
//
// Ordering with the kernels around this one (programmatic dependent launch):
// every thread that reads memory the kernel before may write (xr, by the xr
// producer's copies) or touches the partial sums, counters or y (the
// epilogue) first executes griddepcontrol.wait; the weight copies and the
// decode may run before it. The kernel lets the next one be scheduled as
// soon as it starts, since that one waits in the same way.
// All waits are bounded; a kernel that gives up sets the error flag and exits.
#pragma once

#include "linear_mma.cuh"
#include "rot_block.cuh"

namespace tfx {

namespace {

constexpr int kTcRows = 128;        // row slots of the largest pass (the MMA's N)
constexpr int kTcHalfKt = 8;        // k-tiles per staged half-unit
constexpr int kTcTmemCols = 512;    // accumulators, then the decode warpgroups' A buffers
constexpr int kTcPartialSlots = 3;  // first block, last block, an unshared block

// Shared memory and Tensor Memory of a pass class (SLOTS = 16, 32, 64 or 128
// row slots): a stage holds a half-unit's packed weights and its xr slice for
// SLOTS row slots, so fewer slots make smaller stages and more of them (16 /
// 12 / 8 / 4 at 4 bits).
template <int BITS, int SLOTS, int H>
struct TcCfg {
  static constexpr int kWBytes = 256 * BITS * kTcHalfKt;       // 8 k-tiles x 8 tiles x 32*BITS bytes
  static constexpr int kXrBytes = SLOTS * 16 * kTcHalfKt * 2;  // SLOTS rows x 128 inputs, fp16
  static constexpr int kStageBytes = kWBytes + kXrBytes;
  static constexpr int kStagesFit = (kSmemBudgetWide - 8192 - 2048) / kStageBytes;
  // Decode warpgroups: half-unit q goes to warpgroup q mod kWG. Six (24
  // decode warps, six per SM sub-partition, 64 registers a thread) in the
  // 16-row-slot class at 4, 6 and 8 bits, five up to 32 row slots otherwise,
  // four beyond. Measured on the GB300 (LM head, 1 / 8 / 16 rows): 4 bits
  // 115.6 / 117.5 / 118.1 -> 114.6 / 114.7 / 116.7 us; 6 and 8 bits 1-2 us
  // faster; wkv 6144 -> 25,600 level. At 2, 3 and 5 bits, and at 32 row
  // slots, six were level or slower (wkv 5 bits 42.9 -> 44.9 us).
  static constexpr int kWG = (SLOTS == 16 && (BITS == 4 || BITS == 6 || BITS == 8)) ? 6 : (SLOTS <= 32 ? 5 : 4);
  // A multiple of the warpgroups, so that a stage's previous half-unit went
  // to the same decode warpgroup; and of the half-units of a copy group.
  // The stages hold half-units, but the copies and their barriers go by
  // groups of CG half-units (contiguous in both rings): a whole unit where
  // the ring is deep enough, so that each producer issues one copy a unit;
  // single half-units at 128 row slots, whose ring holds only four.
  static constexpr int kStagesCap = kStagesFit < 16 ? kStagesFit : 16;
  static constexpr int kUnitStep = kWG * H / (kWG % H == 0 ? H : 1);  // lcm(kWG, H) for H in {1, 2}
  static constexpr bool kWholeUnits = kStagesCap / kUnitStep * kUnitStep >= 8;
  static constexpr int kStages = kWholeUnits ? kStagesCap / kUnitStep * kUnitStep : kStagesCap / kWG * kWG;
  static_assert(kStages >= kWG, "one stage per decode warpgroup at least");
  static constexpr int CG = kWholeUnits ? H : 1;
  // The xr ring: kStages, but below two stages per decode warpgroup always a
  // multiple of the chains' period (2 H half-units), so that consecutive
  // uses of an xr slot belong to one chain, i.e. one MMA warp, wherever
  // nothing else orders them: with five slots of single half-units (8 bits,
  // 32 row slots) the MMA warp of half-unit q + 5 could test the slot's
  // barrier before the copy of q (the other chain's) had landed, and a
  // parity wait cannot tell those phases apart. The host simulation of every
  // row-slot class found that schedule.
  static constexpr int kXStages =
      (kStages < 2 * kWG && kStages % (2 * H) != 0) ? (kStages / (2 * H) + 1) * (2 * H) : kStages;
  static constexpr int kUnitSlots = kXStages / CG;  // xr copy slots
  // The weights ring may be deeper than the xr ring: where the wide xr
  // slices leave fewer than two stages per decode warpgroup (6 and 8 bits at
  // 32 and 64 row slots), the weights take the rest of shared memory, a
  // multiple of the warpgroups (and of the copy group) again. Measured on
  // the GB300, LM head: 6 bits, 64 rows 164.8 -> 157.9 us; 8 bits, 32 rows
  // 148.3 -> 132.0 us, 64 rows 166.9 -> 159.7 us. Where the ring already held
  // two stages per warpgroup, a deeper one gained nothing.
  static constexpr int kWStep = kWholeUnits ? kUnitStep : kWG;
  static constexpr int kWFit = (kSmemBudgetWide - 8192 - 2048 - kXStages * kXrBytes) / kWBytes;
  static constexpr int kWCap = kWFit < 24 ? kWFit : 24;
  static constexpr bool kDeepW = kStages < 2 * kWG && CG == H && kWCap / kWStep * kWStep > kStages;
  static constexpr int kWStages = kDeepW ? kWCap / kWStep * kWStep : kStages;
  static constexpr int kWUnitSlots = kWStages / CG;
  static constexpr int kWRingOff = 0;                          // [kWStages][kWBytes]
  static constexpr int kXRingOff = kWStages * kWBytes;         // [kXStages][kXrBytes], 1024-byte aligned
  // Tensor Memory: the accumulators of the two chains (SLOTS columns each),
  // in kAccBufs sets that alternate between segments (so that the MMAs of a
  // segment can start while the epilogue reads the previous one), then one
  // A buffer of 64 columns (8 k-tiles) per decode warpgroup.
  static constexpr int kAccBufs = SLOTS <= 64 ? 2 : 1;
  static constexpr int kACol0 = kAccBufs * 2 * SLOTS;
  static_assert(kACol0 + kWG * 64 <= kTcTmemCols, "Tensor Memory columns");
  // Warp roles: epilogue 0-3, decode 4 .. 4 kWG + 3, weights producer, xr
  // producer, and one MMA warp per chain.
  static constexpr int kProdW = 4 + 4 * kWG;
  static constexpr int kProdX = kProdW + 1;
  static constexpr int kMma = kProdX + 1;  // chain 0; chain 1 is the next warp
  static constexpr int kThreads = (kMma + 2) * 32;
  static constexpr int kXchOff = kXRingOff + kXStages * kXrBytes;
  static constexpr int kBarOff = kXchOff + 8192;
  // wfull, wempty, xfull, xempty per unit slot; afull, aempty per A buffer;
  // dfull, dempty per accumulator set; drain
  // afull: kAFull per warpgroup, its use j on barrier j mod kAFull. A
  // warpgroup's uses go to both chains' MMA warps (at five and six), and a
  // parity wait needs its barrier's previous phase to have been seen by the
  // same waiter: uses j and j + 4 always belong to the same chain.
  static constexpr int kAFull = 4;
  static constexpr int kNumBars = 2 * kWUnitSlots + 2 * kUnitSlots + (kAFull + 1) * kWG + 2 * kAccBufs + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 64;
  static_assert(kBytes <= kSmemBudgetWide, "shared memory");
};

// Decodes k-tile KK of four (strips order) into Tensor Memory at `a_addr`.
template <int BITS, int KK>
__device__ __forceinline__ void tc_decode_kt(const ColQuads<BITS>& cq, int col, uint32_t a_addr) {
  ColWords<BITS> cw;
  quads_to_col_words<BITS, KK>(cq, cw);
  uint32_t a[8];
  decode_col_words<BITS>(cw, col, a);
  tmem_st8(a_addr, a);
}

// Decodes k-tile KK of four (strips order) into registers.
template <int BITS, int KK>
__device__ __forceinline__ void tc_decode_kt_regs(const ColQuads<BITS>& cq, int col, uint32_t (&a)[8]) {
  ColWords<BITS> cw;
  quads_to_col_words<BITS, KK>(cq, cw);
  decode_col_words<BITS>(cw, col, a);
}

// k-tiles of a half-unit a decode warp decodes before it waits for its A
// buffer (held in 8 registers each): two with four decode warpgroups, one
// with five or six (whose threads have 72 or 64 registers).
template <int WG>
constexpr int pre_kt() { return WG >= 5 ? 1 : 2; }

// The pass's row slots: `rows` rounded up to 16 (the MMA's N); slots past
// `rows` read zeros.
__host__ __device__ constexpr int tc_row_slots(int rows) { return (rows + 15) & ~15; }

// A ring position: stage index and the parity of its current phase, advanced
// one half-unit at a time without divisions.
template <int S>
struct RingPos {
  int s = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++s == S) {
      s = 0;
      phase ^= 1u;
    }
  }
};

// The fused rotation's hand-over between CTAs, on three counts in global
// memory: sync[0] hands out (row, 128-block) units, sync[1] counts the units
// rotated, sync[2] the CTAs that are done with both. Units go to whichever
// warps ask first, so CTAs that start late (their SM still held by the
// kernel before) leave the rotation to those already running. In each CTA,
// five actors finish with the counts: the four epilogue warps once a request
// comes back past the last unit, and the xr producer once it has seen every
// unit rotated; `fin` (shared memory, zero at the start) counts them, and
// the CTA's last one counts the CTA into sync[2]. The CTA that completes
// sync[2] sets all three back to zero: no warp of this launch touches them
// after that, and the next launch only after this one has ended (its
// epilogue waits for this kernel first).
__device__ __forceinline__ void rot_cta_done(int* sync, int ctas, int* fin) {
  if (atomicAdd(fin, 1) == 4 && atomicAdd(sync + 2, 1) == ctas - 1) {
    atomicExch(sync, 0);
    atomicExch(sync + 1, 0);
    atomicExch(sync + 2, 0);
  }
}

// One epilogue warp's part of the rotation: asks for units until they run
// out, rotates each into xr, then counts the ones it did into sync[1] (after
// a fence, so that other CTAs that see the count see the rows too).
template <int DT>
__device__ __forceinline__ void rot_claim_units(const MmaParams& p, long long units, int lane, int* fin) {
  const int blocks_per_row = p.in_features >> 7;
  int done = 0;
#pragma unroll 1
  for (;;) {
    long long u = 0;
    if (lane == 0) u = atomicAdd(p.rot_sync, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= units) break;
    rot_block_warp<DT>(p.rot_x, p.rot_suh, p.rot_xr, static_cast<int>(u / blocks_per_row),
                       static_cast<int>(u % blocks_per_row), p.in_features, lane);
    ++done;
  }
  fence_proxy_async_global();
  __syncwarp();
  if (lane == 0) {
    if (done > 0) {
      __threadfence();
      atomicAdd(p.rot_sync + 1, done);
    }
    rot_cta_done(p.rot_sync, p.ctas, fin);
  }
}

// The xr producer's wait: lane 0 polls sync[1] (sleeping between tests,
// bounded by the wait limit of every barrier here) until all `units` are
// rotated; the warp then orders those writes before its tensor copies.
// Returns false, with the abort flag set, if the limit passes.
__device__ __forceinline__ bool rot_wait_all(int* sync, long long units, int ctas, int* fin,
                                             volatile int* abort_flag, int lane) {
  int ok = 1;
  if (lane == 0) {
    const unsigned long long t0 = global_ns();
    while (ld_acquire_gpu(sync + 1) < units) {
      if (*abort_flag || global_ns() - t0 > kWaitLimitNs) {
        ok = 0;
        *abort_flag = 1;
        break;
      }
      __nanosleep(64);
    }
    if (ok) rot_cta_done(sync, ctas, fin);
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  fence_proxy_async_global();  // the rotated rows' generic writes, then this warp's tensor copies of them
  return ok != 0;
}

template <int BITS, int LAYOUT, int UKT, int SLOTS>
__global__ void __launch_bounds__(TcCfg<BITS, SLOTS, UKT / kTcHalfKt>::kThreads, 1)
    trellis_linear_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                             const __grid_constant__ CUtensorMap xmap, const MmaParams p) {
  constexpr int H = UKT / kTcHalfKt;  // half-units per unit
  using T = TcCfg<BITS, SLOTS, H>;
  constexpr int S = T::kXStages;     // xr stages
  constexpr int CG = T::CG;           // half-units per copy
  constexpr int SU = T::kUnitSlots;   // xr copy slots
  constexpr int SW = T::kWStages;     // weights stages
  constexpr int SUW = T::kWUnitSlots;  // weights copy slots
  constexpr int kWG = T::kWG;
  constexpr int kAccB = T::kAccBufs;
  static_assert(SW >= kWG && SW % kWG == 0 && SW % CG == 0, "weights stages must stay with one decode warpgroup");
  static_assert(S % CG == 0, "xr stages");
  extern __shared__ __align__(1024) uint8_t smem[];
  float(*xch)[128] = reinterpret_cast<float(*)[128]>(smem + T::kXchOff);
  const uint32_t bar0 = smem_u32(smem + T::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::kMiscOff);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + T::kMiscOff + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + T::kMiscOff + 8);
  int* rot_fin = reinterpret_cast<int*>(smem + T::kMiscOff + 12);  // the fused rotation's finished actors
  // Barriers of copy slot us (holding half-unit stages us * CG .. + CG - 1).
  auto wfull_bar = [&](int us) { return bar0 + 8u * us; };
  auto wempty_bar = [&](int us) { return bar0 + 8u * (SUW + us); };
  auto xfull_bar = [&](int us) { return bar0 + 8u * (2 * SUW + us); };
  auto xempty_bar = [&](int us) { return bar0 + 8u * (2 * SUW + SU + us); };
  const uint32_t abar0 = bar0 + 8u * (2 * SUW + 2 * SU);
  // A buffer b of chain ch; accumulator set d.
  constexpr int kAF = T::kAFull;
  auto afull_bar = [&](int g, int j) { return abar0 + 8u * (g * kAF + (j & (kAF - 1))); };
  auto aempty_bar = [&](int g) { return abar0 + 8u * (kAF * kWG + g); };
  const uint32_t dbar0 = abar0 + 8u * ((kAF + 1) * kWG);
  auto dfull_bar = [&](int d) { return dbar0 + 8u * d; };
  auto dempty_bar = [&](int d) { return dbar0 + 8u * (kAccB + d); };
  const uint32_t drain = dbar0 + 8u * (2 * kAccB);

  // The warp index through a shuffle from lane 0: the compiler then knows it
  // is the same in every lane, so the roles' loop values live in uniform
  // registers (measured on the GB300: 115.0 -> 111.2 M instructions a launch,
  // 72 -> 70 registers with no spills; LM head 4 bits 118.7 -> 115.6 us).
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const SegmentOrder order(range_start(c, p.units, p.ctas), range_start(c + 1, p.units, p.ctas),
                           p.units_per_block);
  const int n_half = order.n_units * H;
  const int nslots = tc_row_slots(p.rows);
  const uint32_t xr_box_bytes = static_cast<uint32_t>(nslots) * 128;  // 64 inputs x nslots rows

  if (threadIdx.x == 0) {
    // The swizzled B tiles need 1024-byte alignment (their offsets in a stage
    // are multiples of 1024).
    *abort_flag = (smem_u32(smem) & 1023u) != 0 ? 1 : 0;
    *last_flag = 0;
    *rot_fin = 0;
    for (int us = 0; us < SUW; ++us) {
      mbar_init(wfull_bar(us), 1);
      mbar_init(wempty_bar(us), 4 * CG);  // the 4 warps of each half-unit's decoding warpgroup
    }
    for (int us = 0; us < SU; ++us) {
      mbar_init(xfull_bar(us), 1);
      mbar_init(xempty_bar(us), CG);      // the MMAs' commit, per half-unit
    }
    for (int g = 0; g < kWG; ++g) {
      for (int j = 0; j < kAF; ++j) mbar_init(afull_bar(g, j), 4);  // the warpgroup's 4 warps
      mbar_init(aempty_bar(g), 1);                                   // the MMAs' commit
    }
    for (int d = 0; d < kAccB; ++d) {
      mbar_init(dfull_bar(d), 2);  // one signal per chain
      mbar_init(dempty_bar(d), 4);
    }
    mbar_init(drain, 2);
    fence_barrier_init();
  }
  if (warp == T::kMma) {
    tmem_alloc(smem_u32(tmem_holder), kTcTmemCols);
    tmem_relinquish();
  }
  if (warp == T::kProdW && lane == 0 && LAYOUT == kLayoutTiles) tma_prefetch_desc(&wmap);
  if (warp == T::kProdX && lane == 0) tma_prefetch_desc(&xmap);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // The kernel after this one may be scheduled now: every kernel of this
  // library waits (griddepcontrol.wait) for this one before it touches
  // memory this one reads or writes, and only the weights, which no kernel
  // writes, are read before that wait.
  pdl_launch_dependents();

  if (warp == T::kProdW) {
    // ---------------------------------------------------- weights producer
    // One copy per group of CG half-units (contiguous stages). The weights
    // are not written by the kernel before this one, so their copies start
    // at once. The whole warp runs the loop and one elected lane issues the
    // copies, so that their operands are warp-uniform (a loop run by one
    // lane issued several times as many instructions).
    UnitCursor cur(order);
    RingPos<SUW> rp;
    int h0 = 0;  // first half-unit of the group within its unit
    const uint64_t wpolicy = l2_evict_first();  // weights: first out of L2
    int issued = 0;
    const int n_groups = n_half / CG;
    for (int u = 0; u < n_groups; ++u) {
      if (u >= SUW && !__all_sync(0xffffffffu, mbar_wait(wempty_bar(rp.s), rp.phase ^ 1u, abort_flag))) break;
      const uint32_t st = smem_u32(smem + T::kWRingOff + rp.s * CG * T::kWBytes);
      if (elect_one()) {
        mbar_arrive_expect_tx(wfull_bar(rp.s), CG * T::kWBytes);
        if (LAYOUT == kLayoutTiles)
          tma_load_2d(st, &wmap, static_cast<int>(cur.bb) * 32 * BITS, cur.ub() * UKT + h0 * kTcHalfKt,
                      wfull_bar(rp.s), wpolicy);
        else
          bulk_load_1d(st, p.strips + (cur.bb * order.UB + cur.ub()) * (256LL * BITS * UKT) + h0 * T::kWBytes,
                       CG * T::kWBytes, wfull_bar(rp.s), wpolicy);
      }
      __syncwarp();
      issued = u + 1;
      rp.next();
      h0 += CG;
      if (h0 == H) {
        h0 = 0;
        cur.next();
      }
    }
    // Let every copy this warp started land before the CTA can exit.
    for (int u = issued - SUW > 0 ? issued - SUW : 0; u < issued; ++u) {
      volatile int never = 0;
      mbar_wait(wfull_bar(u % SUW), (u / SUW) & 1, &never);
    }
  } else if (warp == T::kProdX) {
    // --------------------------------------------------------- xr producer
    // One copy per group of CG half-units: their 2 CG chunks of 64 inputs.
    pdl_wait_prerequisites();  // xr is written by the kernel before this one
    UnitCursor cur(order);
    RingPos<SU> rp;
    int h0 = 0;
    int issued = 0;
    // With the rotation fused in, xr is written by this launch's CTAs: no
    // copy starts before every share is in (none at all if the wait gives up).
    const bool xr_ready =
        p.rot_x == nullptr ||
        rot_wait_all(p.rot_sync, static_cast<long long>(p.rows) * (p.in_features >> 7), p.ctas, rot_fin,
                     abort_flag, lane);
    const int n_groups = xr_ready ? n_half / CG : 0;
    for (int u = 0; u < n_groups; ++u) {
      if (u >= SU && !__all_sync(0xffffffffu, mbar_wait(xempty_bar(rp.s), rp.phase ^ 1u, abort_flag))) break;
      const uint32_t st = smem_u32(smem + T::kXRingOff + rp.s * CG * T::kXrBytes);
      if (elect_one()) {
        mbar_arrive_expect_tx(xfull_bar(rp.s), 2 * CG * xr_box_bytes);
        tma_load_3d(st, &xmap, 0, 0, cur.ub() * (UKT / 4) + h0 * 2, xfull_bar(rp.s));
      }
      __syncwarp();
      issued = u + 1;
      rp.next();
      h0 += CG;
      if (h0 == H) {
        h0 = 0;
        cur.next();
      }
    }
    for (int u = issued - SU > 0 ? issued - SU : 0; u < issued; ++u) {
      volatile int never = 0;
      mbar_wait(xfull_bar(u % SU), (u / SU) & 1, &never);
    }
  } else if (warp >= 4 && warp < T::kProdW) {
    // -------------------------------------------------------------- decode
    const int wg = (warp - 4) >> 2;              // takes half-units wg, wg + kWG, ...
    const int n = ((warp - 4) & 3) * 32 + lane;  // output of the block = Tensor Memory lane
    const uint32_t lane_off = static_cast<uint32_t>(((warp - 4) & 3) * 32) << 16;
    const int tile = n >> 4, col = n & 15;
    // The warpgroup's A buffer takes its half-units wg, wg + kWG, ... in turn.
    const uint32_t a_addr = tmem + lane_off + T::kACol0 + wg * 64;
    int s = wg;
    uint32_t sphase = 0;
    for (int j = 0;; ++j) {
      const int q = kWG * j + wg;
      if (q >= n_half) break;
      bool ok = mbar_wait(wfull_bar(s / CG), sphase, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;  // tcgen05.st below is warp-collective
      const uint32_t* ws = reinterpret_cast<const uint32_t*>(smem + T::kWRingOff + s * T::kWBytes);
      // The first kPreKt k-tiles are decoded into registers before the A
      // buffer is known to be free (the MMAs of the warpgroup's previous
      // half-unit may still be reading it), then stored once it is.
      constexpr int kPreKt = pre_kt<kWG>();
      uint32_t pre[kPreKt][8];
      if constexpr (LAYOUT == kLayoutTiles) {
#pragma unroll
        for (int kt = 0; kt < kPreKt; ++kt) {
          ColWords<BITS> cw;
          load_col_words<BITS>(ws + (kt * 8 + tile) * 8 * BITS, col, cw);
          decode_col_words<BITS>(cw, col, pre[kt]);
        }
      }
      ColQuads<BITS> cq0;  // strips: the words of k-tiles 0-3, one 128-bit load per word
      if constexpr (LAYOUT == kLayoutStrips) {
        load_col_quads<BITS>(reinterpret_cast<const uint4*>(ws + tile * 32 * BITS), col, cq0);
        tc_decode_kt_regs<BITS, 0>(cq0, col, pre[0]);
        if constexpr (kPreKt > 1) tc_decode_kt_regs<BITS, 1>(cq0, col, pre[kPreKt - 1]);
      }
      // The A buffer: the MMAs of the warpgroup's previous half-unit must be
      // done. (Safe as a parity wait: the warpgroup waited for the MMAs of
      // its half-unit before that one before it stored that one, and the
      // MMAs of this one cannot start before the arrival below, so the
      // barrier is exactly one phase behind or done.)
      if (j >= 1) ok = mbar_wait(aempty_bar(wg), (j - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
#pragma unroll
      for (int kt = 0; kt < kPreKt; ++kt) tmem_st8(a_addr + kt * 8, pre[kt]);
      if constexpr (LAYOUT == kLayoutTiles) {
#pragma unroll
        for (int kt = kPreKt; kt < kTcHalfKt; ++kt) {
          ColWords<BITS> cw;
          load_col_words<BITS>(ws + (kt * 8 + tile) * 8 * BITS, col, cw);
          uint32_t a[8];
          decode_col_words<BITS>(cw, col, a);
          tmem_st8(a_addr + kt * 8, a);
        }
      } else {
        if constexpr (kPreKt < 2) tc_decode_kt<BITS, 1>(cq0, col, a_addr + 1 * 8);
        tc_decode_kt<BITS, 2>(cq0, col, a_addr + 2 * 8);
        tc_decode_kt<BITS, 3>(cq0, col, a_addr + 3 * 8);
        ColQuads<BITS> cq;
        load_col_quads<BITS>(reinterpret_cast<const uint4*>(ws + (8 + tile) * 32 * BITS), col, cq);
        tc_decode_kt<BITS, 0>(cq, col, a_addr + 4 * 8);
        tc_decode_kt<BITS, 1>(cq, col, a_addr + 5 * 8);
        tc_decode_kt<BITS, 2>(cq, col, a_addr + 6 * 8);
        tc_decode_kt<BITS, 3>(cq, col, a_addr + 7 * 8);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(wempty_bar(s / CG));  // the weights of this stage have been read
        mbar_arrive(afull_bar(wg, j));
      }
      s += kWG;
      if (s >= SW) {
        s -= SW;
        sphase ^= 1u;
      }
    }
  } else if (warp == T::kMma || warp == T::kMma + 1) {
    // -------------------------------------------------- MMA, one per chain
    // The whole warp runs the loop and one elected lane issues, so that the
    // operands stay in uniform registers. Each chain's MMAs are issued in
    // input order by its own warp; the two chains' accumulators are
    // independent, so the two warps need no order between them.
    const int ch = warp - T::kMma;  // units at processing positions ch, ch + 2, ...
    const uint32_t idesc = idesc_f16_f32(128, nslots);
    // B descriptors: box 0 (k-tiles 0-3) and box 1 (4-7) of the first
    // stage's xr slice, advanced in 16-byte units.
    // A group's copy lays its 2 CG chunks out back to back (nslots rows of
    // 128 bytes each), so half-unit h of the group in slot us starts at
    // us * CG * kXrBytes + h * 2 * xr_box_bytes of the xr ring.
    const uint64_t bdesc0 = smem_desc_sw128(smem_u32(smem + T::kXRingOff), 1024);
    const uint32_t box_step = xr_box_bytes >> 4;
    const uint32_t unit_step = static_cast<uint32_t>(CG * T::kXrBytes) >> 4;
    bool stop = false;
    for (int sg = 0; sg < order.n_seg && !stop; ++sg) {
      const long long bb = order.block(sg);
      const int seg_lo = order.lo(bb);
      const int P = order.pos(sg, seg_lo);  // the segment's processing positions: [P, P + L)
      const int L = order.hi(bb) - seg_lo;
      const int dset = kAccB == 2 ? (sg & 1) : 0;
      // The accumulator set must have been read out for its previous segment
      // (waited for every segment in order, so no wait skips a phase).
      if (sg >= kAccB) {
        tc_fence_before();
        if (!__all_sync(0xffffffffu, mbar_wait(dempty_bar(dset), ((sg / kAccB) - 1) & 1, abort_flag))) break;
        tc_fence_after();
      }
      const int kf = P + ((ch - P) & 1);  // the chain's first position in the segment
      if (kf >= P + L) {
        // No unit of this chain here (its sum counts as +0): a plain arrival.
        if (lane == 0) mbar_arrive(dfull_bar(dset));
        __syncwarp();
        continue;
      }
      const uint32_t d_addr = tmem + (dset * 2 + ch) * SLOTS;
      // The segment's half-units in groups of B: the MMA warp waits for a
      // whole group, then issues it at once (B = H where one copy brings the
      // whole unit, so one xr wait a unit). Fewer loop passes mean fewer
      // instructions on this warp's sub-partition, which its decode warps pay
      // for. A group never spans two half-units of one warpgroup (B <= 2 <
      // kWG), so no decode waits on MMAs that wait on it.
      constexpr int B = CG == H ? H : 1;
      for (int k = kf; k < P + L && !stop; k += 2) {
#pragma unroll 1
        for (int h0 = 0; h0 < H; h0 += B) {
          int s[B], g[B];  // per half-unit: its stage and the warpgroup that decoded it
          bool ok = true;
#pragma unroll
          for (int i = 0; i < B; ++i) {
            const int q = k * H + h0 + i;
            s[i] = q % S;
            g[i] = q % kWG;
            const int jg = q / kWG;  // its use of that warpgroup's A buffer
            if (i == 0) ok = ok && mbar_wait(xfull_bar(s[i] / CG), (q / S) & 1, abort_flag);
            ok = ok && mbar_wait(afull_bar(g[i], jg), (jg / kAF) & 1, abort_flag);
          }
          if (!__all_sync(0xffffffffu, ok)) {
            stop = true;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int i = 0; i < B; ++i) {
              const uint32_t a_addr = tmem + T::kACol0 + g[i] * 64;
              const uint64_t bd0 = bdesc0 + (s[i] / CG) * unit_step + (s[i] % CG) * 2 * box_step;
              const bool first = k == kf && h0 + i == 0;  // overwrites the accumulator
              // the A buffer and the xr slice are free once these complete
              mma8_commit2(d_addr, a_addr, bd0, bd0 + box_step, idesc, first ? 0u : 1u, aempty_bar(g[i]),
                           xempty_bar(s[i] / CG));
            }
          }
          __syncwarp();
        }
      }
      if (stop) break;
      if (elect_one()) mma_commit(dfull_bar(dset));
      __syncwarp();
    }
    // Every MMA issued must have completed before Tensor Memory is freed.
    if (elect_one()) mma_commit(drain);
    __syncwarp();
  } else if (warp < 4) {
    // ----------------------------------------------------------- epilogue
    pdl_wait_prerequisites();  // partial sums, counters and y follow the kernel before
    if (p.rot_x != nullptr) {
      // The fused rotation: units of the pass's (row, 128-block) units, as
      // many as this warp gets, written to xr.
      const long long nu = static_cast<long long>(p.rows) * (p.in_features >> 7);
      if (p.rot_dtype == 0)
        rot_claim_units<0>(p, nu, lane, rot_fin);
      else if (p.rot_dtype == 1)
        rot_claim_units<1>(p, nu, lane, rot_fin);
      else
        rot_claim_units<2>(p, nu, lane, rot_fin);
    }
    const int t = threadIdx.x;  // output within the block = Tensor Memory lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    LinearPass lp;
    lp.svh = p.svh;
    lp.y = p.y;
    lp.out_dtype = p.out_dtype;
    lp.rows = p.rows;
    lp.in_features = p.in_features;
    lp.out_features = p.out_features;
    const size_t slot_floats = static_cast<size_t>(kTcRows) * 128;
    for (int sg = 0; sg < order.n_seg; ++sg) {
      const int b = static_cast<int>(order.block(sg));
      const int seg_lo = order.lo(b);
      const int seg_hi = order.hi(b);
      const int base = order.pos(sg, seg_lo) - seg_lo;
      // A chain with no unit in this segment contributes +0, as in the
      // decode-row kernel.
      const bool has0 = (seg_hi - seg_lo >= 2) || ((base + seg_lo) % 2 == 0);
      const bool has1 = (seg_hi - seg_lo >= 2) || ((base + seg_lo) % 2 != 0);
      const int dset = kAccB == 2 ? (sg & 1) : 0;
      const bool ok = mbar_wait_sleepy(dfull_bar(dset), (sg / kAccB) & 1, abort_flag, 64);
      if (!group_all(1, 128, ok)) break;  // the named barriers below need all 128 threads
      tc_fence_after();
      // Shared with other CTAs unless this CTA's range holds the whole block
      // (the CTAs that share it are found only then: 64-bit divisions).
      const bool shared = seg_hi - seg_lo != order.UB;
      int c_first = c, c_last = c;
      if (shared) {
        c_first = cta_of_unit(static_cast<long long>(b) * order.UB, p.units, p.ctas);
        c_last = cta_of_unit(static_cast<long long>(b + 1) * order.UB - 1, p.units, p.ctas);
      }
      const int slot = shared ? partial_slot(c, b, p) : 2;
      float* mine = p.partials + (static_cast<size_t>(c) * kTcPartialSlots + slot) * slot_floats;
      if (SLOTS == 16 && !shared) {
        // A block this CTA owns, in a pass of up to 16 rows: the two chains'
        // sum stays in registers, and only the pass's rows are rotated.
        float v[16], g1[16];
        tmem_ld16(tmem + lane_off + (dset * 2) * SLOTS, v);
        tmem_ld16(tmem + lane_off + (dset * 2 + 1) * SLOTS, g1);
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = __fadd_rn(has0 ? v[r] : 0.0f, has1 ? g1[r] : 0.0f);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty_bar(dset));  // the MMA warp may reuse the set
        fwht_outputs(v, p.rows, t, xch, 1, 128);
        store_outputs(v, lp, b, t, 0);
        group_sync(1, 128);
        continue;
      }
      // The two chains' sums, added in chain order, into this CTA's slot.
#pragma unroll 1
      for (int r0 = 0; r0 < p.rows; r0 += 16) {
        float g0[16], g1[16];
        tmem_ld16(tmem + lane_off + (dset * 2) * SLOTS + r0, g0);
        tmem_ld16(tmem + lane_off + (dset * 2 + 1) * SLOTS + r0, g1);
#pragma unroll
        for (int r = 0; r < 16; ++r) mine[(r0 + r) * 128 + t] = __fadd_rn(has0 ? g0[r] : 0.0f, has1 ? g1[r] : 0.0f);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty_bar(dset));  // the MMA warp may reuse the set
      bool finish = true;
      if (shared) {
        __threadfence();
        group_sync(1, 128);
        if (t == 0) {
          const int old = atomicAdd(p.counters + b, 1);
          *last_flag = (old == c_last - c_first) ? 1 : 0;
        }
        group_sync(1, 128);
        finish = *last_flag != 0;
        if (finish) __threadfence();
      } else {
        group_sync(1, 128);
      }
      if (finish) {
#pragma unroll 1
        for (int r0 = 0; r0 < p.rows; r0 += 16) {
          float v[16];
          for (int cc = (shared ? c_first : c); cc <= (shared ? c_last : c); ++cc) {
            const int sl = shared ? partial_slot(cc, b, p) : 2;
            const float* src = p.partials + (static_cast<size_t>(cc) * kTcPartialSlots + sl) * slot_floats;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = __ldcg(src + (r0 + r) * 128 + t);
            const bool first = !shared || cc == c_first;
#pragma unroll
            for (int r = 0; r < 16; ++r) v[r] = first ? x[r] : __fadd_rn(v[r], x[r]);
          }
          // All 16 slots go through the rotation (the ones past `rows` hold
          // zeros): straight-line code, no per-row predicates.
          fwht_outputs(v, 16, t, xch, 1, 128);
          store_outputs(v, lp, b, t, r0);
        }
        if (shared && t == 0) p.counters[b] = 0;
      }
      group_sync(1, 128);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == T::kMma) {
    volatile int never = 0;
    mbar_wait(drain, 0, &never);  // both chains' MMAs have completed
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err_flag, 1);
}

template <int BITS, int LAYOUT, int UKT, int SLOTS>
cudaError_t tc_smem_attr() {
  static PerDeviceOnce<kMaxAttrDevices> once;
  return smem_attr_once(once, trellis_linear_tc_kernel<BITS, LAYOUT, UKT, SLOTS>,
                        TcCfg<BITS, SLOTS, UKT / kTcHalfKt>::kBytes);
}

// Launches the kernel of row-slot class SLOTS.
template <int BITS, int UKT, int SLOTS>
cudaError_t launch_tc(const CUtensorMap& wmap, const CUtensorMap& xmap, const MmaParams& p, bool strips, int ctas,
                      cudaStream_t stream) {
  cudaError_t e = strips ? tc_smem_attr<BITS, kLayoutStrips, UKT, SLOTS>() : tc_smem_attr<BITS, kLayoutTiles, UKT, SLOTS>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(TcCfg<BITS, SLOTS, UKT / kTcHalfKt>::kThreads);
  cfg.dynamicSmemBytes = TcCfg<BITS, SLOTS, UKT / kTcHalfKt>::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return strips ? cudaLaunchKernelEx(&cfg, trellis_linear_tc_kernel<BITS, kLayoutStrips, UKT, SLOTS>, wmap, xmap, p)
                : cudaLaunchKernelEx(&cfg, trellis_linear_tc_kernel<BITS, kLayoutTiles, UKT, SLOTS>, wmap, xmap, p);
}

// One pass of the row-slot class SLOTS: the tensor maps (whose boxes are
// the class's copy groups) and the launch.
template <int BITS, int UKT, int SLOTS>
cudaError_t run_tc_class(const LinearPass& lp, const TcWorkspace& ws, bool strips, cudaStream_t stream) {
  constexpr int CG = TcCfg<BITS, SLOTS, UKT / kTcHalfKt>::CG;
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap wmap, xmap;
  memset(&wmap, 0, sizeof(wmap));
  if (!strips) {
    // Packed weights as rows of u64, one row per k-tile; a box is a copy
    // group: 8 CG k-tiles x 8 tiles.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(lp.out_features) * BITS / 4,
                                static_cast<cuuint64_t>(lp.in_features / 16)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lp.out_features) * BITS * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(32 * BITS), static_cast<cuuint32_t>(kTcHalfKt * CG)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint32_t*>(lp.trellis), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // xr [rows][in] fp16 viewed as (64 inputs, rows, in / 64): a box of
    // (64, the pass's row slots, 2 CG) lands as a copy group's chunks of 64
    // inputs (the MMA's K-major B operand for 4 k-tiles each), each the row
    // slots' 128-byte rows written with the 128-byte swizzle; slots past
    // `rows` are zeros.
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(lp.rows), static_cast<cuuint64_t>(lp.in_features / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(lp.in_features) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(tc_row_slots(lp.rows)), static_cast<cuuint32_t>(2 * CG)};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(lp.xr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  MmaParams p;
  p.strips = reinterpret_cast<const uint8_t*>(lp.trellis);
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
  if (lp.rot_x != nullptr) {
    if (ws.rot_sync == nullptr) return cudaErrorInvalidValue;
    p.rot_x = lp.rot_x;
    p.rot_suh = lp.rot_suh;
    p.rot_xr = const_cast<__half*>(lp.xr);
    p.rot_sync = ws.rot_sync;
    p.rot_dtype = lp.rot_dtype;
  }
  return launch_tc<BITS, UKT, SLOTS>(wmap, xmap, p, strips, ws.ctas, stream);
}

// One pass of up to 128 rows.
template <int BITS, int UKT>
cudaError_t run_tc(const LinearPass& lp, const TcWorkspace& ws, bool strips, cudaStream_t stream) {
  const int ns = tc_row_slots(lp.rows);
  if (ns <= 16) return run_tc_class<BITS, UKT, 16>(lp, ws, strips, stream);
  if (ns <= 32) return run_tc_class<BITS, UKT, 32>(lp, ws, strips, stream);
  if (ns <= 64) return run_tc_class<BITS, UKT, 64>(lp, ws, strips, stream);
  return run_tc_class<BITS, UKT, 128>(lp, ws, strips, stream);
}

}  // namespace
}  // namespace tfx
