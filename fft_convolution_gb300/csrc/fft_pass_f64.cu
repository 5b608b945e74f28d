// fft_pass_f64.cu -- instantiates the HBM pass / 2D column pass kernel for
// double complex data, every supported on-chip length, both directions.
#include "fft_pass_cluster.cuh"

namespace fftgb {

cudaError_t launch_pass_f64(int dir, const PassArgs &a, const void *in, void *out,
                            cudaStream_t st) {
  if (dir < 0) return dispatch_pass<double, -1, kPassMaxLogF64>(a, in, out, st);
  return dispatch_pass<double, +1, kPassMaxLogF64>(a, in, out, st);
}

}  // namespace fftgb
