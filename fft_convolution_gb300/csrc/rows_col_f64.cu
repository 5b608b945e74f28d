// rows_col_f64.cu -- instantiates the row pass with the first column radix
// folded in (fft_rows_col.cuh) for double complex data.
#include "fft_rows_col.cuh"

namespace fftgb {

cudaError_t launch_rows_col_f64(int logw, int logr, int dir, const void *in, void *out, int log_h,
                                long long planes, cudaStream_t st) {
  if (dir < 0) return dispatch_rows_col<double, -1>(logw, logr, in, out, log_h, planes, st);
  return dispatch_rows_col<double, +1>(logw, logr, in, out, log_h, planes, st);
}

}  // namespace fftgb
