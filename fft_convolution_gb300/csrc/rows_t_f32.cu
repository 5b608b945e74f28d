// rows_t_f32.cu -- float instantiations of the row transforms with transposed
// stores (fft_rows_t.cuh).
#include "fft_rows_t.cuh"

namespace fftgb {

cudaError_t launch_rows_t_f32(int logn, int dir, const void *in, void *out, long long rows,
                              int log_r, cudaStream_t st) {
  return dir < 0 ? dispatch_rows_t<float, -1>(logn, in, out, rows, log_r, st)
                 : dispatch_rows_t<float, 1>(logn, in, out, rows, log_r, st);
}

int rows_t_max_log_f32() {
  // Largest length whose transposed-store kernel fits one block (1024
  // threads, 227 KB of shared memory: 4 rows of 4096 floats staged).
  return 12;
}

}  // namespace fftgb
