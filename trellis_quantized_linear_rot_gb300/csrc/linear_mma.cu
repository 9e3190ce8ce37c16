// The trellis linear's launch dispatch: the CTA count and the kernel for the
// bit width (each width's kernels are compiled in their own file,
// linear_mma_w<bits>.cu, from the kernel in linear_mma.cuh).
#include "kernels.h"

namespace tfx {

namespace {

// k-tiles per unit (one rule for the CTA count and the launch): 16 where the
// input count allows it and at least five stages still fit, else 8.
int unit_kt(int in_features, int bits) { return (in_features % 256 == 0 && bits <= 5) ? 16 : 8; }

}  // namespace

int trellis_linear_mma_ctas(int num_sms, int in_features, int out_features, int bits) {
  const long long units =
      static_cast<long long>(out_features / 128) * (in_features / (16 * unit_kt(in_features, bits)));
  return static_cast<int>(units < num_sms ? units : num_sms);
}

cudaError_t launch_trellis_linear_mma(const LinearPass& p, const TcWorkspace& ws, bool strips,
                                      cudaStream_t stream) {
  const int ukt = unit_kt(p.in_features, p.bits);
  switch (p.bits) {
    case 2: return run_trellis_linear_w2(p, ws, strips, ukt, stream);
    case 3: return run_trellis_linear_w3(p, ws, strips, ukt, stream);
    case 4: return run_trellis_linear_w4(p, ws, strips, ukt, stream);
    case 5: return run_trellis_linear_w5(p, ws, strips, ukt, stream);
    case 6: return run_trellis_linear_w6(p, ws, strips, ukt, stream);
    case 8: return run_trellis_linear_w8(p, ws, strips, ukt, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tfx
