// polymul.cu -- integer polynomial multiplication through fp64 transforms
// ("FFT on GPU", polynomial-multiplication section: coefficient form ->
// point values at the roots of unity -> pointwise product -> inverse
// transform -> coefficients).
//
// Both inputs are zero-padded to L = 2^log_len >= na + nb - 1 and
// transformed with the multi-pass Stockham kernel of fft_pass.cuh; the
// padding and the int64 -> fp64 conversion happen inside the first pass's
// loads, the pointwise product inside the last forward pass of b (it reads
// A_k at the position it is about to write), and the 1/L scaling plus the
// rounding to int64 inside the last inverse pass's stores.  No separate
// conversion, product or rounding kernel touches HBM.
#include "fft_pass.cuh"

namespace fftgb {

// int64 coefficients, zero beyond na (the padding), as complex fp64.
struct LoadInt64Pad {
  const long long *a;
  long long na;
  __device__ __forceinline__ double2 operator()(long long b, long long pos) const {
    return pos < na ? make_c<double2>((double)a[b * na + pos], 0.0) : make_c<double2>(0.0, 0.0);
  }
};

// Pointwise product with the other operand's spectrum: out_k = X_k * A_k.
struct StoreMulComplex {
  double2 *out;
  const double2 *other;
  long long bstride;
  __device__ __forceinline__ void operator()(long long b, long long pos, double2 v) const {
    const long long k = b * bstride + pos;
    out[k] = c_mul(v, other[k]);
  }
};

// Real part rounded to the nearest integer (halves away from zero), only
// the first nc coefficients.
struct StoreRoundInt64 {
  long long *c;
  long long nc;
  __device__ __forceinline__ void operator()(long long b, long long pos, double2 v) const {
    if (pos < nc) c[b * nc + pos] = llround(v.x);
  }
};

// Largest on-chip factor used per pass for the fp64 polynomial transforms.
constexpr int kPolyPassLog = 9;

template <int DIR, class Load, class Store, int LOGL = 1>
cudaError_t poly_pass(int log_l, Load load, Store store, int log_n, int log_m, long long batch,
                      cudaStream_t st) {
  if constexpr (LOGL > kPolyPassLog) {
    return cudaErrorInvalidValue;
  } else {
    if (log_l == LOGL)
      return launch_pass_t<double, LOGL, DIR>(load, store, log_n, log_m, /*twiddle=*/1, batch,
                                              st);
    return poly_pass<DIR, Load, Store, LOGL + 1>(log_l, load, store, log_n, log_m, batch, st);
  }
}

cudaError_t launch_polymul(const long long *a, long long na, const long long *b, long long nb,
                           long long *c, long long batch, int log_len, void *scratch,
                           cudaStream_t st) {
  const long long L = 1LL << log_len;
  const long long nc = na + nb - 1;
  double2 *S[3];
  for (int k = 0; k < 3; ++k) S[k] = static_cast<double2 *>(scratch) + (long long)k * batch * L;

  // Split log_len into P nearly equal factors of at most kPolyPassLog bits.
  int P = (log_len + kPolyPassLog - 1) / kPolyPassLog;
  if (P < 1) P = 1;
  int logs[8];
  for (int k = 0; k < P; ++k) logs[k] = log_len / P + (k < log_len % P ? 1 : 0);

  using LC = LoadComplex<double2>;
  using SC = StoreComplex<double2>;
  cudaError_t e = cudaSuccess;

  // Plain complex -> complex passes use the library's fp64 pass kernels.
  auto plain = [&](int dir, int log_l, const double2 *in, double2 *out, int log_m) {
    PassArgs pa{log_len, log_l, log_m, 1, batch};
    return launch_pass_f64(dir, pa, in, out, st);
  };

  // Forward transform of one int64 operand.  Pass k writes S[k % 2] except
  // the last, which goes through `last_store`.
  auto forward = [&](const long long *src, long long nsrc, auto last_store) -> cudaError_t {
    int log_m = 0;
    const double2 *prev = nullptr;
    for (int k = 0; k < P; ++k) {
      const bool first = k == 0, final_pass = k == P - 1;
      cudaError_t r;
      if (first && final_pass)
        r = poly_pass<-1>(logs[k], LoadInt64Pad{src, nsrc}, last_store, log_len, log_m, batch, st);
      else if (first)
        r = poly_pass<-1>(logs[k], LoadInt64Pad{src, nsrc}, SC{S[k % 2], L}, log_len, log_m,
                          batch, st);
      else if (final_pass)
        r = poly_pass<-1>(logs[k], LC{prev, L}, last_store, log_len, log_m, batch, st);
      else
        r = plain(-1, logs[k], prev, S[k % 2], log_m);
      if (r != cudaSuccess) return r;
      prev = S[k % 2];
      log_m += logs[k];
    }
    return cudaSuccess;
  };

  // A = FFT(a) into S[2].
  e = forward(a, na, SC{S[2], L});
  if (e != cudaSuccess) return e;
  // B = FFT(b) * A into S[(P-1) % 2].
  double2 *Bbuf = S[(P - 1) % 2];
  e = forward(b, nb, StoreMulComplex{Bbuf, S[2], L});
  if (e != cudaSuccess) return e;

  // c = round(IFFT(B)); intermediates alternate over the two other buffers.
  int log_m = 0;
  const double2 *prev = Bbuf;
  double2 *other[2] = {S[P % 2], S[2]};
  for (int k = 0; k < P; ++k) {
    const bool final_pass = k == P - 1;
    cudaError_t r;
    if (final_pass)
      r = poly_pass<+1>(logs[k], LC{prev, L}, StoreRoundInt64{c, nc}, log_len, log_m, batch, st);
    else
      r = plain(+1, logs[k], prev, other[k % 2], log_m);
    if (r != cudaSuccess) return r;
    if (!final_pass) prev = other[k % 2];
    log_m += logs[k];
  }
  return cudaSuccess;
}

}  // namespace fftgb
