// real_f64.cu -- double instantiations of the real-sequence transforms (real.cuh).
#include "real.cuh"

namespace fftgb {

cudaError_t launch_real_rows_f64(int logh, int dir, const void *in, void *out, long long batch,
                                 cudaStream_t st) {
  return dir < 0 ? dispatch_real_rows<double, true>(logh, in, out, batch, st)
                 : dispatch_real_rows<double, false>(logh, in, out, batch, st);
}

cudaError_t real_aux_f64(int op, const RealAuxArgs &a, cudaStream_t st) {
  return real_aux_t<double>(op, a, st);
}

}  // namespace fftgb
