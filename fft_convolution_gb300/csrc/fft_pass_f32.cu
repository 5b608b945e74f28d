// fft_pass_f32.cu -- instantiates the HBM pass / 2D column pass kernel for
// float complex data, every supported on-chip length, both directions.
#include "fft_pass.cuh"

namespace fftgb {

cudaError_t launch_pass_f32(int dir, const PassArgs &a, const void *in, void *out,
                            cudaStream_t st) {
  if (dir < 0) return dispatch_pass<float, -1, kPassMaxLogF32>(a, in, out, st);
  return dispatch_pass<float, +1, kPassMaxLogF32>(a, in, out, st);
}

}  // namespace fftgb
