// tf_trellis_linear_noalloc: the trellis linear without any allocation.
//
// tf_trellis_linear allocates a small workspace with cudaMalloc on its first
// call on each device. Some callers cannot allow that: a serving process
// whose caching allocator has already reserved the device memory it plans
// around (a later cudaMalloc can fail or fragment that plan), and code that
// must not hit the implicit device synchronisation that cudaMalloc and
// cudaFree may cause. This entry point instead keeps its scratch (partial
// sums of output blocks shared by two CTAs, one arrival counter per output
// block) in a fixed array in device memory that exists on every GPU that
// loads this library, for as long as the process runs.
#include <cuda_runtime.h>

#include <array>
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "tf_exl3.h"

namespace tfx {

namespace {

// Limits of the fixed scratch array.
constexpr int kNoAllocMaxCtas = 160;          // CTAs of one launch (one per SM)
constexpr int kNoAllocMaxBlocks = 16384;      // output blocks of 128: out_features <= 2,097,152
constexpr size_t kPartialFloats = static_cast<size_t>(kNoAllocMaxCtas) * 2 * 16 * 128;
constexpr size_t kScratchBytes = kPartialFloats * sizeof(float) + kNoAllocMaxBlocks * sizeof(int);

// The scratch array: partial sums ([ctas][2][16][128] fp32), then the
// counters. About 2.6 MB per GPU.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct NoAllocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
std::array<NoAllocDevice, kMaxDevices> g_dev;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace tfx

using namespace tfx;

extern "C" tf_status tf_trellis_linear_noalloc(const void* xr, const void* trellis, const void* svh,
                                               void* y, int out_dtype, int rows, int in_features,
                                               int out_features, int bits, void* stream) {
  // The refusals of tf_trellis_linear first, then the limit of the array.
  if (rows < 0 || in_features <= 0 || in_features % 128 || in_features > (1 << 20) ||
      out_features <= 0 || out_features % 128 || out_features > (1 << 24))
    return TF_ERR_SHAPE;
  if (!(bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8)) return TF_ERR_BITS;
  if (out_dtype != TF_F16 && out_dtype != TF_F32 && out_dtype != TF_BF16) return TF_ERR_DTYPE;
  if (out_features / 128 > kNoAllocMaxBlocks) return TF_ERR_SCRATCH;
  if (rows == 0) return TF_OK;
  if (!xr || !trellis || !svh || !y) return TF_ERR_NULL;
  if (!aligned16(xr) || !aligned16(trellis) || !aligned16(svh) || !aligned16(y)) return TF_ERR_ALIGN;
  int* err_flag = nullptr;
  int num_sms = 0;
  int device = -1;
  tf_status s = current_device_state(&device, &num_sms, &err_flag);
  if (s != TF_OK) return s;
  s = check_pointers_on_device(device, xr, trellis, svh, y);
  if (s != TF_OK) return s;
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    NoAllocDevice& d = g_dev[device];
    if (!d.ready) {
      // The symbol's device address on the current device (the host-side
      // name is only a stand-in and must never reach a kernel).
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess) return record_cuda_error(e, "cudaGetSymbolAddress (no-alloc scratch)");
      d.scratch = static_cast<unsigned char*>(ptr);
      d.ready = true;
    }
    scratch = d.scratch;
  }
  TcWorkspace ws;
  ws.partials = reinterpret_cast<float*>(scratch);
  ws.counters = reinterpret_cast<int*>(scratch + kPartialFloats * sizeof(float));
  ws.err_flag = err_flag;
  ws.partial_floats_per_cta = kMmaPartialFloatsPerCta;  // passes of 16 rows, mma.sync kernel only
  ws.ctas = trellis_linear_mma_ctas(num_sms < kNoAllocMaxCtas ? num_sms : kNoAllocMaxCtas, in_features,
                                    out_features, bits);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t out_elem = out_dtype == TF_F32 ? 4 : 2;
  for (int r0 = 0; r0 < rows; r0 += 16) {
    // The counters must start at zero. A completed launch leaves them at
    // zero, but one that gave up a bounded wait may not, so every pass
    // clears the ones it uses first.
    cudaError_t e =
        cudaMemsetAsync(ws.counters, 0, static_cast<size_t>(out_features / 128) * sizeof(int), st);
    if (e != cudaSuccess) return record_cuda_error(e, "cudaMemsetAsync (no-alloc counters)");
    LinearPass p;
    p.xr = static_cast<const __half*>(xr) + static_cast<size_t>(r0) * in_features;
    p.trellis = static_cast<const uint32_t*>(trellis);
    p.svh = static_cast<const __half*>(svh);
    p.y = static_cast<char*>(y) + static_cast<size_t>(r0) * out_features * out_elem;
    p.out_dtype = out_dtype;
    p.rows = rows - r0 < 16 ? rows - r0 : 16;
    p.in_features = in_features;
    p.out_features = out_features;
    p.bits = bits;
    e = launch_trellis_linear_mma(p, ws, false, st);
    if (e != cudaSuccess) return record_cuda_error(e, "trellis linear (no-alloc) launch");
  }
  return TF_OK;
}
