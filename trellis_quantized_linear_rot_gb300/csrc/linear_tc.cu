// The trellis linear for decode rows on GB300: a persistent, warp-specialised
// kernel with TMA-fed shared-memory stages, decode into Tensor Memory and
// tcgen05 MMAs accumulating in Tensor Memory.
//
// Method: "hip exl3: the input rotation and trellis linear for decode rows",
// section "What this changes" (second bullet): the trellis linear at 2..8 bits
// with mul1, one fp16 fma per decoded weight, each row's K sums in a fixed
// order (so a row's bits do not depend on the rows sharing its launch), no
// split of the sums visible to the caller, no bias; the output rotation and
// svh finish each 128-output block.
//
// Work: the (output block b, 128-input unit) grid, block-major, is cut into
// one contiguous range per CTA (one CTA per SM). A CTA walks its range unit by
// unit. Consecutive units of one block form a segment whose sums accumulate
// in one Tensor Memory buffer in input order. A block whose units all belong
// to one CTA is finished by that CTA; a block cut between CTAs has each CTA
// store its partial sums, and the CTA that arrives last adds them in CTA
// order (the input order) and finishes the block. The cut depends only on the
// shape and the CTA count, never on the rows, so a row's bits are the same in
// every launch on the same device.
//
// Warp roles (NWG decode warpgroups):
//   warps 0-3        epilogue: Tensor Memory -> fp32 sums -> output rotation
//                    -> svh -> y (or partial sums to the workspace)
//   warps 4..4NWG+3  decode: warpgroup g takes units g, g+NWG, ...; thread n
//                    decodes output n of the block for the unit's 8 k-tiles
//                    into Tensor Memory lane n (the MMA's A operand)
//   warp 4NWG+4      producer: one thread issues the TMA copies of each unit
//                    (packed weights of 8 k-tiles x 8 tiles, and the 16 x 128
//                    slice of xr laid out as the MMA's B operand)
//   warp 4NWG+5      MMA: allocates Tensor Memory; one thread issues
//                    tcgen05.mma (M = 128 outputs, N = 16 row slots, K = 16)
// All waits are bounded; a kernel that gives up sets the error flag and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "decode.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace tfx {

namespace {

constexpr int kUnitKt = 8;           // k-tiles per unit (128 inputs)
constexpr int kXrUnitBytes = 4096;   // 8 k-tiles x 16 rows x 16 fp16
constexpr int kSlotsPerWg = 2;       // Tensor Memory A slots per decode warpgroup
constexpr int kSlotCols = 64;        // 8 k-tiles x 8 columns (16 fp16 per lane)
constexpr int kDCols = 16;           // fp32 sums: 16 row slots
constexpr int kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_f16_f32(128, 16);
constexpr int kSmemBudget = 200 * 1024;

#ifndef TF_DECODE_WARPGROUPS
#define TF_DECODE_WARPGROUPS 2
#endif
constexpr int kDecodeWarpgroups = TF_DECODE_WARPGROUPS;  // 2 or 3 (Tensor Memory fits 3)

template <int BITS>
struct Cfg {
  static constexpr int kWUnitBytes = 2048 * BITS;  // 8 k-tiles x 8 tiles x 32*BITS bytes
  static constexpr int kStageBytes = kWUnitBytes + kXrUnitBytes;
  static constexpr int kStagesFit = kSmemBudget / kStageBytes;
  static constexpr int kStages = kStagesFit < 12 ? kStagesFit : 12;
};

struct TcParams {
  const __half* svh;
  void* y;
  float* partials;     // [ctas][2][16][128]
  int* counters;       // [out_features / 128]
  int* err_flag;
  long long units;     // (out/128) * (in/128)
  int units_per_block; // in / 128
  int ctas;
  int out_f32;
  int rows;
  int in_features;
  int out_features;
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
__device__ __forceinline__ int partial_slot(int c, int b, const TcParams& p) {
  const long long first_block = range_start(c, p.units, p.ctas) / p.units_per_block;
  return b == first_block ? 0 : 1;
}

template <int BITS, int NWG>
struct Layout {
  static constexpr int kStages = Cfg<BITS>::kStages;
  static constexpr int kStageBytes = Cfg<BITS>::kStageBytes;
  static constexpr int kXchOff = kStages * kStageBytes;
  static constexpr int kBarOff = kXchOff + 16 * 128 * 4;
  // barriers: full[S], empty[S], a_full[NWG*2], a_empty[NWG*2], d_full[2], d_empty[2], drain
  static constexpr int kNumBars = 2 * kStages + 4 * NWG + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // At least 120 KB, so that two CTAs never share an SM (each takes all of
  // its Tensor Memory) at any width.
  static constexpr int kBytes = kMiscOff + 64 > 120 * 1024 ? kMiscOff + 64 : 120 * 1024;
  static constexpr int kThreads = (6 + 4 * NWG) * 32;
};

template <int BITS, int NWG>
__global__ void __launch_bounds__(Layout<BITS, NWG>::kThreads, 1)
    trellis_linear_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                             const __grid_constant__ CUtensorMap xmap, const TcParams p) {
  using L = Layout<BITS, NWG>;
  constexpr int S = L::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  float(*xch)[128] = reinterpret_cast<float(*)[128]>(smem + L::kXchOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto afull_bar = [&](int g, int k) { return bar0 + 8u * (2 * S + g * 2 + k); };
  auto aempty_bar = [&](int g, int k) { return bar0 + 8u * (2 * S + 2 * NWG + g * 2 + k); };
  auto dfull_bar = [&](int d) { return bar0 + 8u * (2 * S + 4 * NWG + d); };
  auto dempty_bar = [&](int d) { return bar0 + 8u * (2 * S + 4 * NWG + 2 + d); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4 * NWG + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int producer_warp = 4 + 4 * NWG;
  const int mma_warp = producer_warp + 1;
  const int c = blockIdx.x;
  const long long u0 = range_start(c, p.units, p.ctas);
  const long long u1 = range_start(c + 1, p.units, p.ctas);
  const int n_units = static_cast<int>(u1 - u0);
  const int UB = p.units_per_block;
  const long long b_first = u0 / UB;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *last_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 4 + 1);  // the decode warpgroup's 4 warps + the MMA commit
    }
    for (int g = 0; g < NWG; ++g)
      for (int k = 0; k < kSlotsPerWg; ++k) {
        mbar_init(afull_bar(g, k), 4);
        mbar_init(aempty_bar(g, k), 1);
      }
    for (int d = 0; d < 2; ++d) {
      mbar_init(dfull_bar(d), 1);
      mbar_init(dempty_bar(d), 4);
    }
    mbar_init(drain_bar, 1);
    fence_barrier_init();
  }
  if (warp == mma_warp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (warp == producer_warp && lane == 0) {
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t d_col0 = NWG * kSlotsPerWg * kSlotCols;  // D buffers after the A slots

  if (warp == producer_warp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n_units; ++i) {
        const int s = i % S;
        const int k = i / S;
        if (k > 0 && !mbar_wait(empty_bar(s), (k - 1) & 1, abort_flag)) break;
        const long long u = u0 + i;
        const int b = static_cast<int>(u / UB);
        const int ub = static_cast<int>(u % UB);
        const uint32_t st = smem_u32(smem + s * L::kStageBytes);
        mbar_arrive_expect_tx(full_bar(s), L::kStageBytes);
        tma_load_2d(st, &wmap, b * 32 * BITS, ub * kUnitKt, full_bar(s));
        tma_load_3d(st + Cfg<BITS>::kWUnitBytes, &xmap, 0, 0, ub * 16, full_bar(s));
        issued = i + 1;
      }
      // Let every copy this CTA started land before it can exit.
      for (int i = issued - S > 0 ? issued - S : 0; i < issued; ++i) {
        volatile int never = 0;
        mbar_wait(full_bar(i % S), (i / S) & 1, &never);
      }
    }
  } else if (warp == mma_warp) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      for (int i = 0; i < n_units; ++i) {
        const long long u = u0 + i;
        const int b = static_cast<int>(u / UB);
        const int ub = static_cast<int>(u % UB);
        const bool seg_first = (i == 0) || ub == 0;
        const bool seg_last = (i == n_units - 1) || ub == UB - 1;
        const int sg = static_cast<int>(b - b_first);
        const int d = sg & 1;
        const int g = i % NWG;
        const int j = i / NWG;
        const int slot = j % kSlotsPerWg;
        const int ka = j / kSlotsPerWg;
        const int s = i % S;
        if (seg_first && sg >= 2 && !mbar_wait(dempty_bar(d), ((sg >> 1) - 1) & 1, abort_flag)) break;
        if (!mbar_wait(afull_bar(g, slot), ka & 1, abort_flag)) break;
        if (!mbar_wait(full_bar(s), (i / S) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t a_addr = tmem + (g * kSlotsPerWg + slot) * kSlotCols;
        const uint32_t d_addr = tmem + d_col0 + d * kDCols;
        const uint32_t xs = smem_u32(smem + s * L::kStageBytes + Cfg<BITS>::kWUnitBytes);
#pragma unroll
        for (int kt = 0; kt < kUnitKt; ++kt) {
          const uint64_t bdesc = smem_desc_noswizzle(xs + kt * 512, 256, 128);
          mma_f16_tmemA(d_addr, a_addr + kt * 8, bdesc, kIdesc, (seg_first && kt == 0) ? 0u : 1u);
        }
        mma_commit(aempty_bar(g, slot));
        mma_commit(empty_bar(s));
        if (seg_last) mma_commit(dfull_bar(d));
      }
      mma_commit(drain_bar);
      volatile int never = 0;
      mbar_wait(drain_bar, 0, &never);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- decode
    const int g = (warp - 4) >> 2;
    const int t = threadIdx.x - 128 * (g + 1);  // output within the block, 0..127
    const int q = t >> 5;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int tile = t >> 4;
    const int col = t & 15;
    for (int i = g; i < n_units; i += NWG) {
      const int s = i % S;
      const int j = i / NWG;
      const int slot = j % kSlotsPerWg;
      const int ka = j / kSlotsPerWg;
      bool ok = mbar_wait(full_bar(s), (i / S) & 1, abort_flag);
      if (ok && ka > 0) ok = mbar_wait(aempty_bar(g, slot), (ka - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;  // tcgen05.st below is warp-collective
      const uint32_t* wbase =
          reinterpret_cast<const uint32_t*>(smem + s * L::kStageBytes + tile * 32 * BITS);
      const uint32_t a_addr = tmem + lane_off + (g * kSlotsPerWg + slot) * kSlotCols;
      // All loads of the unit first, then the arithmetic of all 8 k-tiles, so
      // that the shared-memory latency is paid once per unit.
      ColWords<BITS> cw[kUnitKt];
#pragma unroll
      for (int kt = 0; kt < kUnitKt; ++kt) load_col_words<BITS>(wbase + kt * 64 * BITS, col, cw[kt]);
#pragma unroll
      for (int kt = 0; kt < kUnitKt; ++kt) {
        uint32_t a[8];
        decode_col_words<BITS>(cw[kt], col, a);
        tmem_st8(a_addr + kt * 8, a);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(afull_bar(g, slot));
        mbar_arrive(empty_bar(s));
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int t = threadIdx.x;  // output within the block, TMEM lane t
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const long long b_last = (u1 - 1) / UB;
    LinearPass lp;
    lp.svh = p.svh;
    lp.y = p.y;
    lp.out_f32 = p.out_f32;
    lp.rows = p.rows;
    lp.in_features = p.in_features;
    lp.out_features = p.out_features;
    for (long long bb = b_first; bb <= b_last; ++bb) {
      const int b = static_cast<int>(bb);
      const int sg = static_cast<int>(bb - b_first);
      const int d = sg & 1;
      const bool ok = mbar_wait(dfull_bar(d), (sg >> 1) & 1, abort_flag);
      if (!group_all(1, 128, ok)) break;  // the group's named barriers need all 128 threads
      tc_fence_after();
      float v[16];
      tmem_ld16(tmem + lane_off + d_col0 + d * kDCols, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty_bar(d));
      const int c_first = cta_of_unit(static_cast<long long>(b) * UB, p.units, p.ctas);
      const int c_last = cta_of_unit(static_cast<long long>(b + 1) * UB - 1, p.units, p.ctas);
      if (c_first == c_last) {
        block_epilogue(v, lp, b, t, xch, 1, 128);
        continue;
      }
      // Block shared with other CTAs: publish the partial sums, count arrivals.
      float* mine = p.partials + (static_cast<size_t>(c) * 2 + partial_slot(c, b, p)) * 16 * 128;
#pragma unroll
      for (int r = 0; r < 16; ++r)
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
              p.partials + (static_cast<size_t>(cc) * 2 + partial_slot(cc, b, p)) * 16 * 128;
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            if (r < p.rows) {
              const float x = __ldcg(src + r * 128 + t);
              v[r] = (cc == c_first) ? x : __fadd_rn(v[r], x);
            }
          }
        }
        block_epilogue(v, lp, b, t, xch, 1, 128);
        if (t == 0) p.counters[b] = 0;
      }
      group_sync(1, 128);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err_flag, 1);
  if (warp == mma_warp) tmem_dealloc(tmem, kTmemCols);
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

template <int BITS, int NWG>
struct TcLauncher {
  static cudaError_t run(const LinearPass& lp, const TcWorkspace& ws, cudaStream_t stream) {
    using L = Layout<BITS, NWG>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
      attr_err = cudaFuncSetAttribute(trellis_linear_tc_kernel<BITS, NWG>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    auto encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;

    CUtensorMap wmap, xmap;
    {
      // Packed weights as rows of u64: one row per k-tile, O * BITS / 4 words.
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(lp.out_features) * BITS / 4,
                                  static_cast<cuuint64_t>(lp.in_features / 16)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lp.out_features) * BITS * 2};
      const cuuint32_t box[2] = {static_cast<cuuint32_t>(32 * BITS), static_cast<cuuint32_t>(kUnitKt)};
      const cuuint32_t estr[2] = {1, 1};
      CUresult r = encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint32_t*>(lp.trellis),
                          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
      // xr as (8 inputs, rows, in / 8): a box of (8, 16, 16) lands as the MMA's
      // B operand for 8 k-tiles: [k / 8][row][k % 8], rows past `rows` zero.
      const cuuint64_t dims[3] = {8, static_cast<cuuint64_t>(lp.rows),
                                  static_cast<cuuint64_t>(lp.in_features / 8)};
      const cuuint64_t strides[2] = {static_cast<cuuint64_t>(lp.in_features) * 2, 16};
      const cuuint32_t box[3] = {8, 16, 16};
      const cuuint32_t estr[3] = {1, 1, 1};
      CUresult r = encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(lp.xr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    TcParams p;
    p.svh = lp.svh;
    p.y = lp.y;
    p.partials = ws.partials;
    p.counters = ws.counters;
    p.err_flag = ws.err_flag;
    p.units_per_block = lp.in_features / 128;
    p.units = static_cast<long long>(lp.out_features / 128) * p.units_per_block;
    p.ctas = ws.ctas;
    p.out_f32 = lp.out_f32;
    p.rows = lp.rows;
    p.in_features = lp.in_features;
    p.out_features = lp.out_features;
    trellis_linear_tc_kernel<BITS, NWG><<<ws.ctas, L::kThreads, L::kBytes, stream>>>(wmap, xmap, p);
    return cudaGetLastError();
  }
};

}  // namespace

int trellis_linear_tc_ctas(int num_sms, int in_features, int out_features) {
  const long long units = static_cast<long long>(out_features / 128) * (in_features / 128);
  return static_cast<int>(units < num_sms ? units : num_sms);
}

cudaError_t launch_trellis_linear_tc(const LinearPass& p, const TcWorkspace& ws, cudaStream_t stream) {
  switch (p.bits) {
    case 2: return TcLauncher<2, kDecodeWarpgroups>::run(p, ws, stream);
    case 3: return TcLauncher<3, kDecodeWarpgroups>::run(p, ws, stream);
    case 4: return TcLauncher<4, kDecodeWarpgroups>::run(p, ws, stream);
    case 5: return TcLauncher<5, kDecodeWarpgroups>::run(p, ws, stream);
    case 6: return TcLauncher<6, kDecodeWarpgroups>::run(p, ws, stream);
    case 8: return TcLauncher<8, kDecodeWarpgroups>::run(p, ws, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tfx
