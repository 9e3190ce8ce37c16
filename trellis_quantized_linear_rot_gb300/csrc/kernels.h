// Internal launchers shared by the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tf_exl3.h"

namespace tfx {

// Host helpers of the C ABI (api.cu) for entry points in other files.
tf_status current_device_state(int* device, int* num_sms, int** err_flag);
tf_status check_pointers_on_device(int device, const void* a, const void* b, const void* c, const void* d);
tf_status record_cuda_error(cudaError_t e, const char* what);

cudaError_t launch_rot_in(const void* x, int x_dtype, const __half* suh, __half* xr, int rows,
                          int in_features, int num_sms, cudaStream_t stream);

cudaError_t launch_trellis_decode(const uint32_t* trellis, __half* w, int in_features,
                                  int out_features, int bits, cudaStream_t stream);

// Rows of one pass of the linear: the weights are decoded once per pass, and
// each decoded tile feeds the MMAs of all the pass's rows. Two kernels give
// every row the same bits: the mma.sync kernel (passes of up to
// kMaxDecodePassRows rows) and the tcgen05 kernel (up to kMaxPassRows).
constexpr int kMaxDecodePassRows = 16;
constexpr int kMaxPassRows = 128;
// Partial sums per CTA: the tcgen05 kernel's [3][128][128] and the mma.sync
// kernel's [2][16][128] fp32. The library's workspaces hold the larger.
constexpr size_t kTcPartialFloatsPerCta = 3 * 128 * 128;
constexpr size_t kMmaPartialFloatsPerCta = 2 * 16 * 128;
constexpr size_t kPartialFloatsPerCta = kTcPartialFloatsPerCta;

// The kernel of a pass: the tcgen05 kernel wherever the workspace holds its
// partial sums; a workspace too small for them (the no-allocation entry
// point's) keeps passes of up to 16 rows on the mma.sync kernel. Both give
// every row the same bits.
inline bool pass_uses_tc(int rows, int bits, bool strips, size_t partial_floats_per_cta) {
  (void)bits;
  (void)strips;
  if (rows > kMaxDecodePassRows) return true;
  return partial_floats_per_cta >= kTcPartialFloatsPerCta;
}

// One pass of at most kMaxPassRows rows through the trellis linear.
struct LinearPass {
  const __half* xr;          // [rows][in] fp16
  const uint32_t* trellis;   // packed tiles
  const __half* svh;         // [out]
  void* y;                   // [rows][out]
  int out_dtype;             // TF_F16, TF_F32 or TF_BF16
  int rows;                  // 1..kMaxPassRows
  int in_features;
  int out_features;
  int bits;
  // The rotation fused into the launch: when rot_x is set, the launch first
  // writes xr = rot_in(rot_x, rot_suh) for its rows (rot_dtype 0 fp16, 1 fp32,
  // 2 bf16) into `xr`, then reads it back for the sums.
  const void* rot_x = nullptr;
  const __half* rot_suh = nullptr;
  int rot_dtype = 0;
};

// Per-device state the linear needs: SM count, error flag, partial-sum
// workspace for output blocks shared by several CTAs.
struct DeviceCtx {
  int device = -1;
  int num_sms = 0;
  int* err_flag = nullptr;       // device int, OR of error bits
  float* partials = nullptr;     // [slots][16][128] fp32
  int* counters = nullptr;       // [max_blocks] arrival counters, then the fused rotation's three
                                 // counts; all kept at zero between calls
  size_t partial_slots = 0;
  size_t counter_len = 0;
};

// Workspace of the persistent linear: partial sums of output blocks cut
// between CTAs ([ctas][2][16][128] fp32) and one arrival counter per output
// block (zero between calls).
struct TcWorkspace {
  float* partials;                // partial sums: room for partial_floats_per_cta fp32 per CTA
  int* counters;
  int* err_flag;
  int ctas;
  size_t partial_floats_per_cta;  // capacity per CTA (picks the kernels it can serve)
  int* rot_sync = nullptr;        // the fused rotation's counts (units handed out, rotated; CTAs done)
};

int trellis_linear_mma_ctas(int num_sms, int in_features, int out_features, int bits);
// The kernels of one bit width, with ukt k-tiles per unit (8 or 16).
cudaError_t run_trellis_linear_w2(const LinearPass& p, const TcWorkspace& ws, bool strips, int ukt, cudaStream_t s);
cudaError_t run_trellis_linear_w3(const LinearPass& p, const TcWorkspace& ws, bool strips, int ukt, cudaStream_t s);
cudaError_t run_trellis_linear_w4(const LinearPass& p, const TcWorkspace& ws, bool strips, int ukt, cudaStream_t s);
cudaError_t run_trellis_linear_w5(const LinearPass& p, const TcWorkspace& ws, bool strips, int ukt, cudaStream_t s);
cudaError_t run_trellis_linear_w6(const LinearPass& p, const TcWorkspace& ws, bool strips, int ukt, cudaStream_t s);
cudaError_t run_trellis_linear_w8(const LinearPass& p, const TcWorkspace& ws, bool strips, int ukt, cudaStream_t s);
// strips = false: packed tiles in k-tile-major order; true: strips order.
cudaError_t launch_trellis_linear_mma(const LinearPass& p, const TcWorkspace& ws, bool strips,
                                      cudaStream_t stream);
// One bounded barrier wait that nothing completes (the failure-path self-test).
cudaError_t launch_stranded_wait(int* err_flag, cudaStream_t stream);
cudaError_t launch_tiles_to_strips(const uint32_t* tiles, uint32_t* strips, int in_features,
                                   int out_features, int bits, cudaStream_t stream);

}  // namespace tfx
