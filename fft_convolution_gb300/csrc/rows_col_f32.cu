// rows_col_f32.cu -- instantiates the row pass with the first column radix
// folded in (fft_rows_col.cuh) for float complex data.
#include "fft_rows_col.cuh"

namespace fftgb {

cudaError_t launch_rows_col_f32(int logw, int logr, int dir, const void *in, void *out, int log_h,
                                long long planes, cudaStream_t st) {
  if (dir < 0) return dispatch_rows_col<float, -1>(logw, logr, in, out, log_h, planes, st);
  return dispatch_rows_col<float, +1>(logw, logr, in, out, log_h, planes, st);
}

}  // namespace fftgb
