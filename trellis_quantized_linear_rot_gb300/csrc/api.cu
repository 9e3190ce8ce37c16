// C ABI of the library (declared in include/tf_exl3.h). Every entry point
// checks its arguments before touching the GPU, then launches on the caller's
// stream. No call allocates per call; the per-device context is created once.
#include <cuda_runtime.h>

#include <array>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "kernels.h"
#include "tf_exl3.h"

namespace tfx {

__device__ int g_device_error;  // OR of error bits set by kernels (1 = a bounded wait gave up)

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxInFeatures = 1 << 20;
constexpr int kMaxOutFeatures = 1 << 24;

thread_local std::string g_last_error;
std::mutex g_ctx_mutex;
std::array<DeviceCtx, kMaxDevices> g_ctx;

tf_status cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return TF_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_bits(int bits) {
  return bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8;
}

bool valid_features(int n, int max) { return n > 0 && n % 128 == 0 && n <= max; }

// Device context of the current device, created on first use.
tf_status current_ctx(DeviceCtx** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    g_last_error = "device index out of range";
    return TF_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_ctx_mutex);
  DeviceCtx& c = g_ctx[dev];
  if (c.device < 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* flag = nullptr;
    e = cudaGetSymbolAddress(&flag, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    c.num_sms = sms;
    c.err_flag = static_cast<int*>(flag);
    c.device = dev;
  }
  *out = &c;
  return TF_OK;
}

// The linear's workspace on the current device: partial sums for up to one
// CTA per SM and one arrival counter per possible output block, allocated
// and zeroed once, on the first call that needs it.
tf_status ensure_workspace(DeviceCtx* c) {
  std::lock_guard<std::mutex> lock(g_ctx_mutex);
  if (c->partials != nullptr) return TF_OK;
  const size_t slots = static_cast<size_t>(c->num_sms);
  const size_t counters = kMaxOutFeatures / 128 + 3;  // + the fused rotation's three counts
  void* part = nullptr;
  void* cnt = nullptr;
  cudaError_t e = cudaMalloc(&part, slots * kPartialFloatsPerCta * sizeof(float));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc (workspace)");
  e = cudaMalloc(&cnt, counters * sizeof(int));
  if (e != cudaSuccess) {
    cudaFree(part);
    return cuda_fail(e, "cudaMalloc (workspace)");
  }
  e = cudaMemset(cnt, 0, counters * sizeof(int));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(part);
    cudaFree(cnt);
    return cuda_fail(e, "cudaMemset (workspace)");
  }
  c->partials = static_cast<float*>(part);
  c->counters = static_cast<int*>(cnt);
  c->partial_slots = slots;
  c->counter_len = counters;
  return TF_OK;
}

// The pointer must be device (or managed) memory of `device`.
tf_status check_device_ptr(const void* p, int device) {
  cudaPointerAttributes attr;
  std::memset(&attr, 0, sizeof(attr));
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TF_ERR_POINTER;
  }
  if ((attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) &&
      attr.device == device)
    return TF_OK;
  return TF_ERR_POINTER;
}

template <typename... P>
tf_status check_device_ptrs(int device, P... ptrs) {
  for (const void* p : {static_cast<const void*>(ptrs)...}) {
    tf_status s = check_device_ptr(p, device);
    if (s != TF_OK) return s;
  }
  return TF_OK;
}

}  // namespace

tf_status current_device_state(int* device, int* num_sms, int** err_flag) {
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  *device = ctx->device;
  *num_sms = ctx->num_sms;
  *err_flag = ctx->err_flag;
  return TF_OK;
}

tf_status check_pointers_on_device(int device, const void* a, const void* b, const void* c, const void* d) {
  return check_device_ptrs(device, a, b, c, d);
}

tf_status record_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }

}  // namespace tfx

using namespace tfx;

extern "C" {

int tf_abi_version(void) { return 1; }

const char* tf_status_string(int status) {
  switch (status) {
    case TF_OK: return "ok";
    case TF_ERR_NULL: return "a required pointer is NULL";
    case TF_ERR_SHAPE: return "unsupported shape (rows < 0, or features not positive multiples of 128)";
    case TF_ERR_BITS: return "bits must be 2, 3, 4, 5, 6 or 8";
    case TF_ERR_DTYPE: return "unsupported dtype code";
    case TF_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case TF_ERR_CUDA: return "a CUDA call failed (see tf_last_error)";
    case TF_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case TF_ERR_POINTER: return "a pointer is not device memory of the current device";
    case TF_ERR_SCRATCH: return "the problem needs more scratch than the given workspace or the fixed no-allocation array holds";
    default: return "unknown status";
  }
}

const char* tf_last_error(void) { return g_last_error.c_str(); }

size_t tf_trellis_bytes(int in_features, int out_features, int bits) {
  if (!valid_features(in_features, kMaxInFeatures) || !valid_features(out_features, kMaxOutFeatures) ||
      !valid_bits(bits))
    return 0;
  return static_cast<size_t>(in_features) * static_cast<size_t>(out_features) * bits / 8;
}

tf_status tf_rot_in(const void* x, int x_dtype, const void* suh, void* xr, int rows,
                    int in_features, void* stream) {
  if (rows < 0 || !valid_features(in_features, kMaxInFeatures)) return TF_ERR_SHAPE;
  if (x_dtype != TF_F16 && x_dtype != TF_F32 && x_dtype != TF_BF16) return TF_ERR_DTYPE;
  if (rows == 0) return TF_OK;
  if (!x || !suh || !xr) return TF_ERR_NULL;
  if (!aligned16(x) || !aligned16(suh) || !aligned16(xr)) return TF_ERR_ALIGN;
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  s = check_device_ptrs(ctx->device, x, suh, xr);
  if (s != TF_OK) return s;
  const int dt = x_dtype == TF_F16 ? 0 : (x_dtype == TF_F32 ? 1 : 2);
  cudaError_t e = launch_rot_in(x, dt, static_cast<const __half*>(suh), static_cast<__half*>(xr),
                                rows, in_features, ctx->num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rot_in launch");
  return TF_OK;
}

static tf_status linear_entry(const void* xr, const void* trellis, const void* svh, void* y,
                              int out_dtype, int rows, int in_features, int out_features, int bits,
                              bool strips, void* stream) {
  if (rows < 0 || !valid_features(in_features, kMaxInFeatures) ||
      !valid_features(out_features, kMaxOutFeatures))
    return TF_ERR_SHAPE;
  if (!valid_bits(bits)) return TF_ERR_BITS;
  if (out_dtype != TF_F16 && out_dtype != TF_F32 && out_dtype != TF_BF16) return TF_ERR_DTYPE;
  if (rows == 0) return TF_OK;
  if (!xr || !trellis || !svh || !y) return TF_ERR_NULL;
  if (!aligned16(xr) || !aligned16(trellis) || !aligned16(svh) || !aligned16(y)) return TF_ERR_ALIGN;
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  s = check_device_ptrs(ctx->device, xr, trellis, svh, y);
  if (s != TF_OK) return s;
  s = ensure_workspace(ctx);
  if (s != TF_OK) return s;
  TcWorkspace ws;
  ws.partials = ctx->partials;
  ws.counters = ctx->counters;
  ws.err_flag = ctx->err_flag;
  ws.ctas = trellis_linear_mma_ctas(ctx->num_sms, in_features, out_features, bits);
  ws.partial_floats_per_cta = kPartialFloatsPerCta;
  const size_t out_elem = out_dtype == TF_F32 ? 4 : 2;
  for (int r0 = 0; r0 < rows; r0 += kMaxPassRows) {
    LinearPass p;
    p.xr = static_cast<const __half*>(xr) + static_cast<size_t>(r0) * in_features;
    p.trellis = static_cast<const uint32_t*>(trellis);
    p.svh = static_cast<const __half*>(svh);
    p.y = static_cast<char*>(y) + static_cast<size_t>(r0) * out_features * out_elem;
    p.out_dtype = out_dtype;
    p.rows = rows - r0 < kMaxPassRows ? rows - r0 : kMaxPassRows;
    p.in_features = in_features;
    p.out_features = out_features;
    p.bits = bits;
    cudaError_t e = launch_trellis_linear_mma(p, ws, strips, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "trellis linear launch");
  }
  return TF_OK;
}

static tf_status rot_in_linear_entry(const void* x, int x_dtype, const void* suh, void* xr,
                                     const void* trellis, const void* svh, void* y, int out_dtype, int rows,
                                     int in_features, int out_features, int bits, bool strips, void* stream) {
  if (rows < 0 || !valid_features(in_features, kMaxInFeatures) ||
      !valid_features(out_features, kMaxOutFeatures))
    return TF_ERR_SHAPE;
  if (!valid_bits(bits)) return TF_ERR_BITS;
  if (x_dtype != TF_F16 && x_dtype != TF_F32 && x_dtype != TF_BF16) return TF_ERR_DTYPE;
  if (out_dtype != TF_F16 && out_dtype != TF_F32 && out_dtype != TF_BF16) return TF_ERR_DTYPE;
  if (rows == 0) return TF_OK;
  if (!x || !suh || !xr || !trellis || !svh || !y) return TF_ERR_NULL;
  if (!aligned16(x) || !aligned16(suh) || !aligned16(xr) || !aligned16(trellis) || !aligned16(svh) ||
      !aligned16(y))
    return TF_ERR_ALIGN;
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  s = check_device_ptrs(ctx->device, x, suh, xr, trellis, svh, y);
  if (s != TF_OK) return s;
  s = ensure_workspace(ctx);
  if (s != TF_OK) return s;
  TcWorkspace ws;
  ws.partials = ctx->partials;
  ws.counters = ctx->counters;
  ws.err_flag = ctx->err_flag;
  ws.ctas = trellis_linear_mma_ctas(ctx->num_sms, in_features, out_features, bits);
  ws.partial_floats_per_cta = kPartialFloatsPerCta;
  ws.rot_sync = ctx->counters + (ctx->counter_len - 3);
  const size_t x_elem = x_dtype == TF_F32 ? 4 : 2;
  const size_t out_elem = out_dtype == TF_F32 ? 4 : 2;
  const int dt = x_dtype == TF_F16 ? 0 : (x_dtype == TF_F32 ? 1 : 2);
  for (int r0 = 0; r0 < rows; r0 += kMaxPassRows) {
    LinearPass p;
    p.xr = static_cast<const __half*>(xr) + static_cast<size_t>(r0) * in_features;
    p.trellis = static_cast<const uint32_t*>(trellis);
    p.svh = static_cast<const __half*>(svh);
    p.y = static_cast<char*>(y) + static_cast<size_t>(r0) * out_features * out_elem;
    p.out_dtype = out_dtype;
    p.rows = rows - r0 < kMaxPassRows ? rows - r0 : kMaxPassRows;
    p.in_features = in_features;
    p.out_features = out_features;
    p.bits = bits;
    p.rot_x = static_cast<const char*>(x) + static_cast<size_t>(r0) * in_features * x_elem;
    p.rot_suh = static_cast<const __half*>(suh);
    p.rot_dtype = dt;
    cudaError_t e = launch_trellis_linear_mma(p, ws, strips, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fused rot_in + trellis linear launch");
  }
  return TF_OK;
}

tf_status tf_rot_in_linear(const void* x, int x_dtype, const void* suh, void* xr, const void* trellis,
                           const void* svh, void* y, int out_dtype, int rows, int in_features,
                           int out_features, int bits, void* stream) {
  return rot_in_linear_entry(x, x_dtype, suh, xr, trellis, svh, y, out_dtype, rows, in_features,
                             out_features, bits, false, stream);
}

tf_status tf_rot_in_linear_strips(const void* x, int x_dtype, const void* suh, void* xr,
                                  const void* strips, const void* svh, void* y, int out_dtype, int rows,
                                  int in_features, int out_features, int bits, void* stream) {
  return rot_in_linear_entry(x, x_dtype, suh, xr, strips, svh, y, out_dtype, rows, in_features,
                             out_features, bits, true, stream);
}

tf_status tf_trellis_linear(const void* xr, const void* trellis, const void* svh, void* y,
                            int out_dtype, int rows, int in_features, int out_features, int bits,
                            void* stream) {
  return linear_entry(xr, trellis, svh, y, out_dtype, rows, in_features, out_features, bits, false,
                      stream);
}

tf_status tf_trellis_linear_strips(const void* xr, const void* strips, const void* svh, void* y,
                                   int out_dtype, int rows, int in_features, int out_features,
                                   int bits, void* stream) {
  return linear_entry(xr, strips, svh, y, out_dtype, rows, in_features, out_features, bits, true,
                      stream);
}

// Caller workspace of tf_trellis_linear_ws: partial sums for every CTA of a
// launch (kPartialFloatsPerCta fp32 each), then one arrival counter per
// output block, each part starting on a 256-byte boundary.
static size_t ws_partial_bytes(int ctas) {
  const size_t b = static_cast<size_t>(ctas) * kPartialFloatsPerCta * sizeof(float);
  return (b + 255) & ~static_cast<size_t>(255);
}

size_t tf_trellis_workspace_bytes(int in_features, int out_features, int bits) {
  if (!valid_features(in_features, kMaxInFeatures) || !valid_features(out_features, kMaxOutFeatures) ||
      !valid_bits(bits))
    return 0;
  DeviceCtx* ctx = nullptr;
  if (current_ctx(&ctx) != TF_OK) return 0;
  const int ctas = trellis_linear_mma_ctas(ctx->num_sms, in_features, out_features, bits);
  return ws_partial_bytes(ctas) + static_cast<size_t>(out_features / 128) * sizeof(int);
}

tf_status tf_trellis_linear_ws(const void* xr, const void* trellis, const void* svh, void* y, int out_dtype,
                               int rows, int in_features, int out_features, int bits, int layout,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (rows < 0 || !valid_features(in_features, kMaxInFeatures) ||
      !valid_features(out_features, kMaxOutFeatures) || (layout != 0 && layout != 1))
    return TF_ERR_SHAPE;
  if (!valid_bits(bits)) return TF_ERR_BITS;
  if (out_dtype != TF_F16 && out_dtype != TF_F32 && out_dtype != TF_BF16) return TF_ERR_DTYPE;
  if (rows == 0) return TF_OK;
  if (!xr || !trellis || !svh || !y || !workspace) return TF_ERR_NULL;
  if (!aligned16(xr) || !aligned16(trellis) || !aligned16(svh) || !aligned16(y) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return TF_ERR_ALIGN;
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  s = check_device_ptrs(ctx->device, xr, trellis, svh, y, workspace);
  if (s != TF_OK) return s;
  TcWorkspace ws;
  ws.ctas = trellis_linear_mma_ctas(ctx->num_sms, in_features, out_features, bits);
  ws.partial_floats_per_cta = kPartialFloatsPerCta;
  const size_t part = ws_partial_bytes(ws.ctas);
  if (workspace_bytes < part + static_cast<size_t>(out_features / 128) * sizeof(int)) return TF_ERR_SCRATCH;
  ws.partials = static_cast<float*>(workspace);
  ws.counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + part);
  ws.err_flag = ctx->err_flag;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The counters must start at zero; clear the ones this call uses on its stream.
  cudaError_t e = cudaMemsetAsync(ws.counters, 0, static_cast<size_t>(out_features / 128) * sizeof(int), st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (workspace counters)");
  const size_t out_elem = out_dtype == TF_F32 ? 4 : 2;
  for (int r0 = 0; r0 < rows; r0 += kMaxPassRows) {
    LinearPass p;
    p.xr = static_cast<const __half*>(xr) + static_cast<size_t>(r0) * in_features;
    p.trellis = static_cast<const uint32_t*>(trellis);
    p.svh = static_cast<const __half*>(svh);
    p.y = static_cast<char*>(y) + static_cast<size_t>(r0) * out_features * out_elem;
    p.out_dtype = out_dtype;
    p.rows = rows - r0 < kMaxPassRows ? rows - r0 : kMaxPassRows;
    p.in_features = in_features;
    p.out_features = out_features;
    p.bits = bits;
    e = launch_trellis_linear_mma(p, ws, layout == 1, st);
    if (e != cudaSuccess) return cuda_fail(e, "trellis linear (caller workspace) launch");
  }
  return TF_OK;
}

tf_status tf_trellis_to_strips(const void* tiles, void* strips, int in_features, int out_features,
                               int bits, void* stream) {
  if (!valid_features(in_features, kMaxInFeatures) || !valid_features(out_features, kMaxOutFeatures))
    return TF_ERR_SHAPE;
  if (!valid_bits(bits)) return TF_ERR_BITS;
  if (!tiles || !strips) return TF_ERR_NULL;
  if (!aligned16(tiles) || !aligned16(strips)) return TF_ERR_ALIGN;
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  s = check_device_ptrs(ctx->device, tiles, strips);
  if (s != TF_OK) return s;
  cudaError_t e = launch_tiles_to_strips(static_cast<const uint32_t*>(tiles), static_cast<uint32_t*>(strips),
                                         in_features, out_features, bits, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tiles-to-strips launch");
  return TF_OK;
}

tf_status tf_trellis_decode(const void* trellis, void* w, int in_features, int out_features,
                            int bits, void* stream) {
  if (!valid_features(in_features, kMaxInFeatures) || !valid_features(out_features, kMaxOutFeatures))
    return TF_ERR_SHAPE;
  if (!valid_bits(bits)) return TF_ERR_BITS;
  if (!trellis || !w) return TF_ERR_NULL;
  if (!aligned16(trellis) || !aligned16(w)) return TF_ERR_ALIGN;
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  s = check_device_ptrs(ctx->device, trellis, w);
  if (s != TF_OK) return s;
  cudaError_t e = launch_trellis_decode(static_cast<const uint32_t*>(trellis), static_cast<__half*>(w),
                                        in_features, out_features, bits,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "trellis decode launch");
  return TF_OK;
}

tf_status tf_selftest_stranded_wait(void* stream) {
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  cudaError_t e = launch_stranded_wait(ctx->err_flag, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stranded-wait self-test launch");
  return TF_OK;
}

tf_status tf_device_error(void* stream) {
  DeviceCtx* ctx = nullptr;
  tf_status s = current_ctx(&ctx);
  if (s != TF_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int flag = 0;
  e = cudaMemcpyFromSymbol(&flag, g_device_error, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (flag != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    if (e == cudaSuccess && ctx->counters != nullptr)
      e = cudaMemset(ctx->counters, 0, ctx->counter_len * sizeof(int));  // an aborted launch may leave counts
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "resetting the error record");
    return TF_ERR_TIMEOUT;
  }
  return TF_OK;
}

}  // extern "C"
