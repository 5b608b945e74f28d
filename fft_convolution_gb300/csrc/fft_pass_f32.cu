// fft_pass_f32.cu -- instantiates the HBM pass / 2D column pass kernel for
// float complex data, every supported on-chip length, both directions.
#include "fft_pass_cluster.cuh"

namespace fftgb {

cudaError_t launch_pass_f32(int dir, const PassArgs &a, const void *in, void *out,
                            cudaStream_t st) {
  if (dir < 0) return dispatch_pass<float, -1, kPassMaxLogF32>(a, in, out, st);
  return dispatch_pass<float, +1, kPassMaxLogF32>(a, in, out, st);
}

namespace {
template <int LOGL = 1> int tile_cols(int log_l) {
  if constexpr (LOGL > kPassMaxLogF32) {
    return 0;
  } else {
    if (log_l == LOGL) return PassConfig<float, LOGL>::C;
    return tile_cols<LOGL + 1>(log_l);
  }
}
}  // namespace

int pass_tile_cols_f32(int log_l) { return tile_cols(log_l); }

}  // namespace fftgb
