// mixed_f64.cu -- double instantiation of the mixed-radix on-chip transforms (mixed.cuh).
#include "mixed.cuh"

namespace fftgb {

cudaError_t mixed_exec_f64(const void *in, void *out, long long batch, const MixedStages &ms,
                           const void *tw, int dir, cudaStream_t st) {
  return mixed_exec_t<double>(in, out, batch, ms, tw, dir, st);
}

}  // namespace fftgb
