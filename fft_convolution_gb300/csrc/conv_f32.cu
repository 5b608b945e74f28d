// conv_f32.cu -- fp32 instantiations of the signal convolution (conv.cuh),
// plus its host-side sizing helpers.
#include "conv.cuh"

namespace fftgb {

size_t convolve_scratch_bytes(long long batch, int h_per_row, int kind, int dtype, int log_len) {
  const size_t elem = dtype == 0 ? 8 : 16;
  const size_t L = (size_t)1 << log_len;
  const size_t trows = kind == CONV_REAL_PAIRS ? (size_t)(batch + 1) / 2 : (size_t)batch;
  const size_t nfilt = h_per_row ? (size_t)batch : 1;
  const int max_on_chip = dtype == 0 ? RowsMaxLog<float>::value : RowsMaxLog<double>::value;
  if (log_len <= max_on_chip) return nfilt * L * elem;
  return (nfilt + 2 * trows) * L * elem;
}

int convolve_num_kernels(int kind, int dtype, int log_len) {
  (void)kind;
  const int max_on_chip = dtype == 0 ? RowsMaxLog<float>::value : RowsMaxLog<double>::value;
  if (log_len <= max_on_chip) return 2;
  int logs[8];
  const int P = conv_split(log_len, dtype == 0 ? conv_pass_log<float>() : conv_pass_log<double>(),
                           logs);
  return 3 * P;
}

int convolve_passes(int dtype, int log_len) {
  int logs[8];
  return conv_split(log_len, dtype == 0 ? conv_pass_log<float>() : conv_pass_log<double>(), logs);
}

cudaError_t launch_convolve_f32(const void *x, long long nx, const void *h, long long nh, void *y,
                                long long batch, int h_per_row, int kind, int log_len,
                                void *scratch, cudaStream_t st) {
  if (kind == CONV_COMPLEX)
    return convolve_t<float, CONV_COMPLEX>(x, nx, h, nh, y, batch, h_per_row, log_len, scratch,
                                           st);
  if (kind == CONV_REAL_PAIRS)
    return convolve_t<float, CONV_REAL_PAIRS>(x, nx, h, nh, y, batch, h_per_row, log_len,
                                              scratch, st);
  return convolve_t<float, CONV_REAL_SINGLE>(x, nx, h, nh, y, batch, h_per_row, log_len,
                                             scratch, st);
}

cudaError_t launch_convolve(const void *x, long long nx, const void *h, long long nh, void *y,
                            long long batch, int h_per_row, int kind, int dtype, int log_len,
                            void *scratch, cudaStream_t st) {
  return dtype == 0 ? launch_convolve_f32(x, nx, h, nh, y, batch, h_per_row, kind, log_len,
                                          scratch, st)
                    : launch_convolve_f64(x, nx, h, nh, y, batch, h_per_row, kind, log_len,
                                          scratch, st);
}

}  // namespace fftgb
