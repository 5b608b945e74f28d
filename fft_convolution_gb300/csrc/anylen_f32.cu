// anylen_f32.cu -- float instantiations of the any-length transforms
// (anylen.cuh): the direct DFT for short lengths and Bluestein.
#include "anylen.cuh"

namespace fftgb {

cudaError_t bluestein_prepare_f32(long long N, int log_m, int dir, void *w, void *B, void *ws,
                                 cudaStream_t st) {
  using V = vec2_t<float>;
  BluesteinState<float> s{static_cast<V *>(w), static_cast<V *>(B), static_cast<V *>(ws)};
  return bluestein_prepare_t<float>(N, log_m, dir, s, st);
}

cudaError_t bluestein_exec_f32(const void *in, void *out, long long N, long long batch, int log_m,
                              double scale, void *w, void *B, void *ws, cudaStream_t st) {
  using V = vec2_t<float>;
  BluesteinState<float> s{static_cast<V *>(w), static_cast<V *>(B), static_cast<V *>(ws)};
  return bluestein_exec_t<float>(in, out, N, batch, log_m, (float)scale, s, st);
}

cudaError_t dft_small_f32(const void *in, void *out, int N, long long batch, int dir, double scale,
                         cudaStream_t st) {
  return dft_small_t<float>(in, out, N, batch, dir, (float)scale, st);
}

}  // namespace fftgb
