// fft_pass_f32.cu -- instantiates the HBM pass / 2D column pass kernel for
// float complex data, every supported on-chip length, both directions.
#include "fft_pass_cluster.cuh"

namespace fftgb {

cudaError_t launch_pass_f32(int dir, const PassArgs &a, const void *in, void *out,
                            cudaStream_t st) {
  if (dir < 0) return dispatch_pass<float, -1, kPassMaxLogF32>(a, in, out, st);
  return dispatch_pass<float, +1, kPassMaxLogF32>(a, in, out, st);
}

// Test hook: one in-place pass of on-chip length 2^13 over 2^15 points (one
// tile, one cluster of 8 blocks) in which block 1's tile load never
// completes; every wait gives up after `polls` polls.
cudaError_t debug_cluster_timeout_f32(void *data, unsigned polls, cudaStream_t st) {
  return launch_pass_cluster_t<float, 13, -1>(data, data, 15, 0, 1, 1, st, 2, polls);
}

}  // namespace fftgb
