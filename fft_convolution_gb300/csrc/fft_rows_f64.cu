// fft_rows_f64.cu -- instantiates the on-chip batched transform for double
// complex data, every supported length, both directions.
#include "fft_rows.cuh"

namespace fftgb {

cudaError_t launch_rows_f64(int logn, int dir, const void *in, void *out, long long batch,
                            cudaStream_t st) {
  if (dir < 0) return dispatch_rows<double, -1>(logn, in, out, batch, st);
  return dispatch_rows<double, +1>(logn, in, out, batch, st);
}

}  // namespace fftgb
