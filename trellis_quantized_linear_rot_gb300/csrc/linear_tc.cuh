// The trellis linear for passes of up to 128 rows on GB300 (prompts, and the
// decode passes the mma.sync kernel is slower at):
// tcgen05 MMAs with the decoded weights in Tensor Memory, the same results
// bit for bit as the decode-row kernel (linear_mma.cuh).
//
// Method: "hip exl3: the input rotation and trellis linear for decode rows",
// section "Known limits": the prompt path follows, registered bit-equal to
// the decode linear. Bit-equality holds because every output element goes
// through the same sums as in the decode-row kernel: the same cut of the
// (block, unit) grid between CTAs, the same two chains per segment (the units
// at even and at odd processing positions, each a chain of K = 16 tensor-core
// steps in input order), their fp32 sum in that order, and the partial sums
// of a shared block added in CTA order. A tcgen05.mma (M = 128, K = 16, A in
// Tensor Memory) gives the same bits as mma.sync.m16n8k16 for the same
// operands and accumulator, also when the 16 inputs of a step are presented
// in another order (checked on the GB300 over 81,920 outputs of chains of
// eight steps with wide exponent ranges).
//
// Per CTA (one per SM): the MMA's M is the 128 outputs of a block (Tensor
// Memory lanes), N the pass's row slots (rows rounded up to 16, at most 128),
// K 16 inputs per k-tile.
// Warp roles:
//   warps 0-3   epilogue: per segment, the two chains' sums from Tensor
//               Memory, added, written to this CTA's partial-sum slot, then
//               (when the CTA owns the block, or arrives last) the output
//               rotation, svh and the stores
//   warps 4-15  decode: three warpgroups (passes of up to 64 row slots;
//               warps 4-19, four warpgroups, at 128) take half-units (8
//               k-tiles) in turn;
//               thread n decodes output n's 16 weights of each k-tile into
//               Tensor Memory lane n (the MMA's A operand)
//   next warp   producer: the copies of each half-unit into a ring of
//               stages sized by the pass's row-slot class (packed weights, and
//               the xr slice of the pass's row slots: two tensor copies of
//               64 inputs x N rows with the 128-byte swizzle, which is the
//               MMA's K-major B layout)
//   last warp   MMA: allocates Tensor Memory; the warp runs the MMA loop and
//               one elected lane issues
// All waits are bounded; a kernel that gives up sets the error flag and exits.
#pragma once

#include "linear_mma.cuh"

namespace tfx {

namespace {

constexpr int kTcRows = 128;     // row slots of a pass (the MMA's N)
constexpr int kTcHalfKt = 8;     // k-tiles per staged half-unit
constexpr int kTcTmemCols = 512;  // acc[2] at columns 0 and 128; one A buffer per warpgroup at 256 + 64 wg
constexpr int kTcPartialSlots = 3;  // first block, last block, an unshared block

// Shared memory of a pass class: stages of a half-unit's packed weights and
// its xr slice for up to SLOTS row slots (32, 64 or 128). Fewer slots make
// smaller stages and so more of them in flight: 12 / 9 / 4 at 4 bits (the
// copies of a stage take longer to land than a warpgroup takes to decode
// one half-unit, so a warpgroup needs stages beyond the one it decodes).
template <int BITS, int SLOTS>
struct TcCfg {
  static constexpr int kWBytes = 256 * BITS * kTcHalfKt;       // 8 k-tiles x 8 tiles x 32*BITS bytes
  static constexpr int kXrBytes = SLOTS * 16 * kTcHalfKt * 2;  // up to SLOTS rows x 128 inputs, fp16
  static constexpr int kStageBytes = kWBytes + kXrBytes;
  static constexpr int kStagesFit = (kSmemBudgetWide - 8192 - 2048) / kStageBytes;
  // A multiple of the warpgroups, so that a stage's previous half-unit went
  // to the same decode warpgroup.
  // Decode warpgroups: three up to 64 row slots, where the decode warps
  // mostly wait and fewer of them leave the MMA and producer warps more issue
  // slots and more stages fit; four at 128 slots (measured at 4 and 6 bits).
  static constexpr int kWG = SLOTS <= 64 ? 3 : 4;
  static constexpr int kProducer = 4 + 4 * kWG;  // warp roles: epilogue 0-3, decode, producer, MMA
  static constexpr int kMma = kProducer + 1;
  static constexpr int kThreads = (kMma + 1) * 32;
  static constexpr int kStages = (kStagesFit < 12 ? kStagesFit : 12) / kWG * kWG;
  static constexpr int kXchOff = kStages * kStageBytes;
  static constexpr int kBarOff = kXchOff + 8192;
  static constexpr int kNumBars = 2 * kStages + 2 * kWG + 3;  // full, empty, afull, aempty, dfull, dempty, drain
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 64;
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

// The pass's row slots: `rows` rounded up to 16 (the MMA's N); slots past
// `rows` read zeros.
__host__ __device__ constexpr int tc_row_slots(int rows) { return (rows + 15) & ~15; }

template <int BITS, int LAYOUT, int UKT, int SLOTS>
__global__ void __launch_bounds__(TcCfg<BITS, SLOTS>::kThreads, 1)
    trellis_linear_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                             const __grid_constant__ CUtensorMap xmap, const MmaParams p) {
  using T = TcCfg<BITS, SLOTS>;
  constexpr int S = T::kStages;
  constexpr int H = UKT / kTcHalfKt;  // half-units per unit
  constexpr int kTcWG = T::kWG;
  constexpr int kTcProducer = T::kProducer;
  constexpr int kTcMma = T::kMma;
  static_assert(S >= kTcWG && S % kTcWG == 0, "stages must stay with one decode warpgroup");
  extern __shared__ __align__(1024) uint8_t smem[];
  float(*xch)[128] = reinterpret_cast<float(*)[128]>(smem + T::kXchOff);
  const uint32_t bar0 = smem_u32(smem + T::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::kMiscOff);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + T::kMiscOff + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + T::kMiscOff + 8);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto afull_bar = [&](int w) { return bar0 + 8u * (2 * S + w); };
  auto aempty_bar = [&](int w) { return bar0 + 8u * (2 * S + kTcWG + w); };
  const uint32_t dfull = bar0 + 8u * (2 * S + 2 * kTcWG);
  const uint32_t dempty = bar0 + 8u * (2 * S + 2 * kTcWG + 1);
  const uint32_t drain = bar0 + 8u * (2 * S + 2 * kTcWG + 2);

  const int warp = threadIdx.x >> 5;
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
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 4 + 1);  // the decoding warpgroup's 4 warps and the MMA thread
    }
    for (int w = 0; w < kTcWG; ++w) {
      mbar_init(afull_bar(w), 4);
      mbar_init(aempty_bar(w), 1);
    }
    mbar_init(dfull, 1);
    mbar_init(dempty, 4);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == kTcMma) {
    tmem_alloc(smem_u32(tmem_holder), kTcTmemCols);
    tmem_relinquish();
  }
  if (warp == kTcProducer && lane == 0) {
    if (LAYOUT == kLayoutTiles) tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kTcProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      pdl_wait_prerequisites();
      UnitCursor cur(order);
      int issued = 0;
      for (int q = 0; q < n_half; ++q) {
        const int s = q % S;
        // A plain wait: the refill of a stage is on the decode warps' path.
        if (q >= S && !mbar_wait(empty_bar(s), ((q / S) - 1) & 1, abort_flag)) break;
        const int h = q % H;
        const int kt0 = cur.ub() * UKT + h * kTcHalfKt;  // first k-tile of the half-unit
        const uint32_t st = smem_u32(smem + s * T::kStageBytes);
        mbar_arrive_expect_tx(full_bar(s), T::kWBytes + 2 * xr_box_bytes);
        if (LAYOUT == kLayoutTiles)
          tma_load_2d(st, &wmap, static_cast<int>(cur.bb) * 32 * BITS, kt0, full_bar(s));
        else
          bulk_load_1d(st, p.strips + (cur.bb * order.UB + cur.ub()) * (256LL * BITS * UKT) + h * T::kWBytes,
                       T::kWBytes, full_bar(s));
        tma_load_2d(st + T::kWBytes, &xmap, kt0 * 16, 0, full_bar(s));
        tma_load_2d(st + T::kWBytes + xr_box_bytes, &xmap, kt0 * 16 + 64, 0, full_bar(s));
        issued = q + 1;
        if (h == H - 1) cur.next();
      }
      for (int q = issued - S > 0 ? issued - S : 0; q < issued; ++q) {
        volatile int never = 0;
        mbar_wait(full_bar(q % S), (q / S) & 1, &never);
      }
    }
  } else if (warp >= 4 && warp < kTcProducer) {
    // -------------------------------------------------------------- decode
    const int wg = (warp - 4) >> 2;           // takes half-units wg, wg + kTcWG, ...
    const int n = ((warp - 4) & 3) * 32 + lane;  // output of the block = Tensor Memory lane
    const uint32_t lane_off = static_cast<uint32_t>(((warp - 4) & 3) * 32) << 16;
    const int tile = n >> 4, col = n & 15;
    for (int j = 0;; ++j) {
      const int q = kTcWG * j + wg;
      if (q >= n_half) break;
      const int s = q % S;
      bool ok = mbar_wait(full_bar(s), (q / S) & 1, abort_flag);
      if (ok && j >= 1) ok = mbar_wait(aempty_bar(wg), (j - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;  // tcgen05.st below is warp-collective
      const uint32_t* ws = reinterpret_cast<const uint32_t*>(smem + s * T::kStageBytes);
      const uint32_t a_addr = tmem + lane_off + 256 + wg * 64;
      if constexpr (LAYOUT == kLayoutTiles) {
#pragma unroll
        for (int kt = 0; kt < kTcHalfKt; ++kt) {
          ColWords<BITS> cw;
          load_col_words<BITS>(ws + (kt * 8 + tile) * 8 * BITS, col, cw);
          uint32_t a[8];
          decode_col_words<BITS>(cw, col, a);
          tmem_st8(a_addr + kt * 8, a);
        }
      } else {
        // Strips: one 128-bit load per word brings it for four k-tiles.
#pragma unroll
        for (int c4 = 0; c4 < kTcHalfKt / 4; ++c4) {
          ColQuads<BITS> cq;
          load_col_quads<BITS>(reinterpret_cast<const uint4*>(ws + (c4 * 8 + tile) * 32 * BITS), col, cq);
          tc_decode_kt<BITS, 0>(cq, col, a_addr + (4 * c4 + 0) * 8);
          tc_decode_kt<BITS, 1>(cq, col, a_addr + (4 * c4 + 1) * 8);
          tc_decode_kt<BITS, 2>(cq, col, a_addr + (4 * c4 + 2) * 8);
          tc_decode_kt<BITS, 3>(cq, col, a_addr + (4 * c4 + 3) * 8);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(afull_bar(wg));
        mbar_arrive(empty_bar(s));
      }
    }
  } else if (warp == kTcMma) {
    // ----------------------------------------------------------------- MMA
    // The whole warp runs the loop and one elected lane issues, so that the
    // operands stay in uniform registers: issued from a lone lane, each MMA
    // costs more than its tensor-core time at these sizes.
    const uint32_t idesc = idesc_f16_f32(128, nslots);
    // B descriptors: the first stage's xr slice, advanced in 16-byte units.
    const uint64_t bdesc0 = smem_desc_sw128(smem_u32(smem + T::kWBytes), 1024);
    const uint32_t box_step = xr_box_bytes >> 4;
    const uint32_t stage_step = static_cast<uint32_t>(T::kStageBytes) >> 4;
    bool stop = false;
    for (int sg = 0; sg < order.n_seg && !stop; ++sg) {
      const long long bb = order.block(sg);
      const int seg_lo = order.lo(bb);
      const int seg_hi = order.hi(bb);
      const int base = order.pos(sg, seg_lo) - seg_lo;  // processing position of unit i: base + i
      // The accumulators must have been read out for the previous segment.
      if (sg >= 1) {
        tc_fence_before();
        if (!__all_sync(0xffffffffu, mbar_wait(dempty, (sg - 1) & 1, abort_flag))) break;
        tc_fence_after();
      }
      uint32_t started = 0;  // bit g: chain g has had its first step
      for (int i = seg_lo; i < seg_hi && !stop; ++i) {
        const int k = base + i;
        const int g = k & 1;  // the chain: units at even / odd processing positions
        const uint32_t d_addr = tmem + g * 128;
        for (int h = 0; h < H; ++h) {
          const int q = k * H + h;
          const int s = q % S;
          const int wg = q % kTcWG, j = q / kTcWG;
          bool ok = mbar_wait(full_bar(s), (q / S) & 1, abort_flag);
          ok = ok && mbar_wait(afull_bar(wg), j & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = tmem + 256 + wg * 64;
          const uint64_t bd = bdesc0 + s * stage_step;
          const uint32_t acc0 = (started >> g) & 1u;
          if (elect_one()) {
#pragma unroll
            for (int kt = 0; kt < kTcHalfKt; ++kt) {
              // B: k-tile kt is inputs 16 (kt % 4) .. + 15 of the swizzled
              // tile kt / 4 (rows of 128 bytes, 8-row groups 1024 apart).
              mma_f16_tmemA(d_addr, a_addr + kt * 8, bd + (kt >> 2) * box_step + (kt & 3) * 2, idesc,
                            kt > 0 ? 1u : acc0);
            }
            mma_commit(aempty_bar(wg));
            mma_commit(empty_bar(s));
          }
          __syncwarp();
          started |= 1u << g;
        }
      }
      if (elect_one()) mma_commit(dfull);
      __syncwarp();
    }
    // Every MMA issued must have completed before Tensor Memory is freed.
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    volatile int never = 0;
    mbar_wait(drain, 0, &never);
  } else {
    // ----------------------------------------------------------- epilogue
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
      const bool ok = mbar_wait_sleepy(dfull, sg & 1, abort_flag, 200);
      if (!group_all(1, 128, ok)) break;  // the named barriers below need all 128 threads
      tc_fence_after();
      const int c_first = cta_of_unit(static_cast<long long>(b) * order.UB, p.units, p.ctas);
      const int c_last = cta_of_unit(static_cast<long long>(b + 1) * order.UB - 1, p.units, p.ctas);
      const bool shared = c_first != c_last;
      const int slot = shared ? partial_slot(c, b, p) : 2;
      float* mine = p.partials + (static_cast<size_t>(c) * kTcPartialSlots + slot) * slot_floats;
      // The two chains' sums, added in chain order, into this CTA's slot.
#pragma unroll 1
      for (int r0 = 0; r0 < p.rows; r0 += 16) {
        float g0[16], g1[16];
        tmem_ld16(tmem + lane_off + r0, g0);
        tmem_ld16(tmem + lane_off + 128 + r0, g1);
#pragma unroll
        for (int r = 0; r < 16; ++r) mine[(r0 + r) * 128 + t] = __fadd_rn(has0 ? g0[r] : 0.0f, has1 ? g1[r] : 0.0f);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty);  // the MMA thread may start the next segment
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
  if (warp == kTcMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err_flag, 1);
}

template <int BITS, int LAYOUT, int UKT, int SLOTS>
cudaError_t tc_smem_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(trellis_linear_tc_kernel<BITS, LAYOUT, UKT, SLOTS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<BITS, SLOTS>::kBytes);
  });
  return err;
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
  cfg.blockDim = dim3(TcCfg<BITS, SLOTS>::kThreads);
  cfg.dynamicSmemBytes = TcCfg<BITS, SLOTS>::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return strips ? cudaLaunchKernelEx(&cfg, trellis_linear_tc_kernel<BITS, kLayoutStrips, UKT, SLOTS>, wmap, xmap, p)
                : cudaLaunchKernelEx(&cfg, trellis_linear_tc_kernel<BITS, kLayoutTiles, UKT, SLOTS>, wmap, xmap, p);
}

// One pass of up to 128 rows.
template <int BITS, int UKT>
cudaError_t run_tc(const LinearPass& lp, const TcWorkspace& ws, bool strips, cudaStream_t stream) {
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap wmap, xmap;
  memset(&wmap, 0, sizeof(wmap));
  if (!strips) {
    // Packed weights as rows of u64, one row per k-tile; a box is 8 k-tiles x 8 tiles.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(lp.out_features) * BITS / 4,
                                static_cast<cuuint64_t>(lp.in_features / 16)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lp.out_features) * BITS * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(32 * BITS), static_cast<cuuint32_t>(kTcHalfKt)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint32_t*>(lp.trellis), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // xr [rows][in] fp16; a box is 64 inputs (128 bytes) x the pass's row
    // slots, written with the 128-byte swizzle: the MMA's K-major B operand
    // for 4 k-tiles. Slots past `rows` are filled with zeros.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(lp.in_features), static_cast<cuuint64_t>(lp.rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lp.in_features) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(tc_row_slots(lp.rows))};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(lp.xr), dims, strides, box,
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
  const int ns = tc_row_slots(lp.rows);
  if (ns <= 32) return launch_tc<BITS, UKT, 32>(wmap, xmap, p, strips, ws.ctas, stream);
  if (ns <= 64) return launch_tc<BITS, UKT, 64>(wmap, xmap, p, strips, ws.ctas, stream);
  return launch_tc<BITS, UKT, 128>(wmap, xmap, p, strips, ws.ctas, stream);
}

}  // namespace
}  // namespace tfx
