// The trellis linear's kernels at 5 bits per weight (one translation unit
// per width so that the widths compile in parallel).
#include "linear_tc.cuh"

namespace tfx {

cudaError_t run_trellis_linear_w5(const LinearPass& p, const TcWorkspace& ws, bool strips, int ukt,
                                  cudaStream_t stream) {
  if (pass_uses_tc(p.rows, 5, strips, ws.partial_floats_per_cta))
    return ukt == 16 ? run_tc<5, 16>(p, ws, strips, stream) : run_tc<5, 8>(p, ws, strips, stream);
  if (p.rows > kMaxDecodePassRows) return cudaErrorInvalidValue;
  return ukt == 16 ? run_mma<5, 16>(p, ws, strips, stream) : run_mma<5, 8>(p, ws, strips, stream);
}

}  // namespace tfx
