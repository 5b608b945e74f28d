// conv_f64.cu -- fp64 instantiations of the signal convolution (conv.cuh).
#include "conv.cuh"

namespace fftgb {

cudaError_t launch_convolve_f64(const void *x, long long nx, const void *h, long long nh, void *y,
                                long long batch, int h_per_row, int kind, int log_len,
                                void *scratch, cudaStream_t st) {
  if (kind == CONV_COMPLEX)
    return convolve_t<double, CONV_COMPLEX>(x, nx, h, nh, y, batch, h_per_row, log_len, scratch,
                                            st);
  if (kind == CONV_REAL_PAIRS)
    return convolve_t<double, CONV_REAL_PAIRS>(x, nx, h, nh, y, batch, h_per_row, log_len,
                                               scratch, st);
  return convolve_t<double, CONV_REAL_SINGLE>(x, nx, h, nh, y, batch, h_per_row, log_len,
                                              scratch, st);
}

}  // namespace fftgb
