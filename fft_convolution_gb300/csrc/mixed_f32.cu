// mixed_f32.cu -- float instantiation of the mixed-radix on-chip transforms (mixed.cuh).
#include "mixed.cuh"

namespace fftgb {

cudaError_t mixed_exec_f32(const void *in, void *out, long long batch, const MixedStages &ms,
                           const void *tw, int dir, cudaStream_t st) {
  return mixed_exec_t<float>(in, out, batch, ms, tw, dir, st);
}

}  // namespace fftgb
