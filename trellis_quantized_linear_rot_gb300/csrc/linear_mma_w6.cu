// The trellis linear's kernels at 6 bits per weight (one translation unit
// per width so that the widths compile in parallel).
#include "linear_tc.cuh"

namespace tfx {

cudaError_t run_trellis_linear_w6(const LinearPass& p, const TcWorkspace& ws, bool strips, int ukt,
                                  cudaStream_t stream) {
  // Units of 8 k-tiles at this width (16 only up to 5 bits).
  if (ukt != 8) return cudaErrorInvalidValue;
  if (pass_uses_tc(p.rows, 6, strips, ws.partial_floats_per_cta)) return run_tc<6, 8>(p, ws, strips, stream);
  if (p.rows > kMaxDecodePassRows) return cudaErrorInvalidValue;
  return run_mma<6, 8>(p, ws, strips, stream);
}

}  // namespace tfx
