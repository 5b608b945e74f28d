// polymul.cu -- integer polynomial multiplication through fp64 transforms
// ("FFT on GPU", polynomial-multiplication section: coefficient form ->
// point values at the roots of unity -> pointwise product -> inverse
// transform -> coefficients).
//
// Both inputs are real, and so is the product, which lets one complex
// transform of length L carry both inputs and one of length L/2 carry the
// product back (both identities follow from the DFT definition and the
// symmetry X_{L-k} = conj(X_k) of a real sequence's spectrum):
//
//  1. z = a + i b, zero-padded to L = 2^log_len >= na + nb - 1; Z = FFT_L(z)
//     (the int64 -> fp64 conversion and the padding happen in the first
//     pass's loads).
//  2. combine (in the loads of the inverse's first pass), for k < L/2:
//        A_k = (Z_k + conj Z_{L-k}) / 2,   B_k = (Z_k - conj Z_{L-k}) / (2i)
//        C_k = A_k B_k  (the pointwise product of the point values),
//     and the same at k + L/2; then
//        E_k = (C_k + C_{k+L/2}) / 2,  O_k = (C_k - C_{k+L/2}) W_L^{-k} / 2,
//        Y_k = E_k + i O_k,
//     which is the L/2-point DFT of y[n] = c[2n] + i c[2n+1].
//  3. y = IFFT_{L/2}(Y) (1/(L/2) folded into its passes); its last pass
//     rounds to int64 and stores c[2n] = Re y[n], c[2n+1] = Im y[n].
//
// The transforms are the multi-pass Stockham kernels of fft_pass.cuh.
#include "fft_pass.cuh"

namespace fftgb {

// a + i b as complex fp64, zero beyond na / nb (the padding).
struct LoadPairInt64 {
  const long long *a;
  const long long *b;
  long long na, nb;
  __device__ __forceinline__ double2 operator()(long long p, long long pos) const {
    return make_c<double2>(pos < na ? (double)a[p * na + pos] : 0.0,
                           pos < nb ? (double)b[p * nb + pos] : 0.0);
  }
};

// y[n] -> c[2n] = round(Re y[n]), c[2n+1] = round(Im y[n]) (halves away from
// zero), only the first nc coefficients.
struct StoreRoundPairsInt64 {
  long long *c;
  long long nc;
  __device__ __forceinline__ void operator()(long long p, long long pos, double2 v) const {
    const long long k = 2 * pos;
    if (k < nc) c[p * nc + k] = llround(v.x);
    if (k + 1 < nc) c[p * nc + k + 1] = llround(v.y);
  }
};

// W_L^{+k} = T_hi[k >> lb] * T_lo[k & (2^lb - 1)] for k < L/2: two short
// tables instead of one sincospi per element.
__global__ void poly_twiddle_tables(double2 *lo, int n_lo, double2 *hi, int n_hi, int lb,
                                    int log_len) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < n_lo) lo[j] = twiddle<+1>((long long)j, log_len, 0.0);
  if (j < n_hi) hi[j] = twiddle<+1>((long long)j << lb, log_len, 0.0);
}

// Y_k (step 2) formed inside the first inverse pass's loads: the point-value
// product of the two packed spectra and the even/odd packing read Z_k,
// Z_{L-k}, Z_{k+L/2} and Z_{L/2-k} straight from the forward transform's
// output, so the product never makes its own trip through HBM.
struct LoadCombine {
  const double2 *Z;
  const double2 *tw_lo, *tw_hi;  // W_L^{-k} = tw_hi[k >> lb] tw_lo[k & (2^lb - 1)]
  int lb;
  long long L;
  __device__ __forceinline__ double2 operator()(long long p, long long k) const {
    const long long H = L >> 1;
    const double2 *z = Z + p * L;
    const double2 zk = z[k], zmk = z[(L - k) & (L - 1)];
    const double2 zh = z[k + H], zmh = z[H - k];
    // A B = (u + conj w)(u - conj w) / (2i) / 2 = (u^2 - conj(w)^2) (-i/4) with
    // u = Z_k, w = Z_{L-k}; returned halved (C/2), the factor E and O need.
    auto half_product = [](double2 u, double2 w) {
      const double re = u.x * u.y + w.x * w.y;                              // Im(u^2 - conj(w)^2) / 2
      const double im = (u.x * u.x - u.y * u.y) - (w.x * w.x - w.y * w.y);  // Re(...)
      return make_c<double2>(0.25 * re, -0.125 * im);
    };
    const double2 Ck = half_product(zk, zmk), Ch = half_product(zh, zmh);  // C/2
    const double2 w = c_mul(tw_hi[k >> lb], tw_lo[k & ((1LL << lb) - 1)]);  // W_L^{-k}
    const double2 O = c_mul(c_sub(Ck, Ch), w);                               // O_k
    return make_c<double2>(Ck.x + Ch.x - O.y, Ck.y + Ch.y + O.x);            // E_k + i O_k
  }
};

// Inter-pass twiddle tables W_{2^log_lm}^e (direction dir) for e < 2^log_lm.
__global__ void poly_pass_tables(double2 *lo, int lo_bits, double2 *hi, int log_lm, int dir) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int n_lo = 1 << lo_bits, n_hi = 1 << (log_lm - lo_bits);
  if (dir < 0) {
    if (j < n_lo) lo[j] = twiddle<-1>((long long)j, log_lm, 0.0);
    if (j < n_hi) hi[j] = twiddle<-1>((long long)j << lo_bits, log_lm, 0.0);
  } else {
    if (j < n_lo) lo[j] = twiddle<+1>((long long)j, log_lm, 0.0);
    if (j < n_hi) hi[j] = twiddle<+1>((long long)j << lo_bits, log_lm, 0.0);
  }
}

// Largest on-chip factor used per pass for the fp64 polynomial transforms.
constexpr int kPolyPassLog = 11;

template <int DIR, class Load, class Store, int LOGL = 1>
cudaError_t poly_pass(int log_l, Load load, Store store, int log_n, int log_m, long long batch,
                      cudaStream_t st, TwiddleTables<double2> tt) {
  if constexpr (LOGL > kPolyPassLog) {
    return cudaErrorInvalidValue;
  } else {
    if (log_l == LOGL)
      return launch_pass_t<double, LOGL, DIR>(load, store, log_n, log_m, /*twiddle=*/1, batch,
                                              st, tt);
    return poly_pass<DIR, Load, Store, LOGL + 1>(log_l, load, store, log_n, log_m, batch, st,
                                                 tt);
  }
}

// Split log_len into nearly equal factors of at most kPolyPassLog bits.
static int split_passes(int log_len, int *logs) {
  int P = (log_len + kPolyPassLog - 1) / kPolyPassLog;
  if (P < 1) P = 1;
  for (int k = 0; k < P; ++k) logs[k] = log_len / P + (k < log_len % P ? 1 : 0);
  return P;
}

// Two buffers of batch * L complex doubles plus the twiddle tables: two
// two-level tables of the inter-pass twiddles (forward, length L; inverse,
// length L/2) and one of W_L^{-k} for the combine step -- six tables of at
// most 2^ceil(log_len/2) entries each.
static long long table_stride(int log_len) { return 1LL << ((log_len + 1) / 2); }

size_t polymul_scratch_bytes(long long batch, int log_len) {
  const size_t L = (size_t)1 << log_len;
  return (2 * (size_t)batch * L + 6 * (size_t)table_stride(log_len)) * sizeof(double2);
}

cudaError_t launch_polymul(const long long *a, long long na, const long long *b, long long nb,
                           long long *c, long long batch, int log_len, void *scratch,
                           cudaStream_t st) {
  if (log_len < 2 || log_len > 27) return cudaErrorInvalidValue;
  const long long L = 1LL << log_len, H = L >> 1;
  const long long nc = na + nb - 1;
  double2 *R[2] = {static_cast<double2 *>(scratch),
                   static_cast<double2 *>(scratch) + batch * L};
  double2 *tables = R[1] + batch * L;
  const long long ts = table_stride(log_len);
  double2 *tw_lo = tables, *tw_hi = tables + ts;                 // combine
  double2 *f_lo = tables + 2 * ts, *f_hi = tables + 3 * ts;      // forward passes
  double2 *i_lo = tables + 4 * ts, *i_hi = tables + 5 * ts;      // inverse passes
  const int lb = log_len / 2;  // k < L/2 splits into lb low bits and log_len-1-lb high bits
  const int n_lo = 1 << lb, n_hi = 1 << (log_len - 1 - lb);
  const int f_bits = (log_len + 1) / 2, i_bits = log_len / 2;

  using LC = LoadComplex<double2>;
  using SC = StoreComplex<double2>;
  cudaError_t e;

  // Twiddle tables (a few thousand sincospi in all).
  {
    const int blocks = (int)(ts / 256) + 1;
    poly_twiddle_tables<<<blocks, 256, 0, st>>>(tw_lo, n_lo, tw_hi, n_hi, lb, log_len);
    poly_pass_tables<<<blocks, 256, 0, st>>>(f_lo, f_bits, f_hi, log_len, -1);
    poly_pass_tables<<<blocks, 256, 0, st>>>(i_lo, i_bits, i_hi, log_len - 1, +1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const TwiddleTables<double2> ftt{f_lo, f_hi, f_bits, log_len},
      itt{i_lo, i_hi, i_bits, log_len - 1};

  // 1. Z = FFT_L(a + i b): pass k writes R[k % 2].
  int logs[8];
  const int P = split_passes(log_len, logs);
  int log_m = 0;
  for (int k = 0; k < P; ++k) {
    SC dst{R[k % 2], L};
    if (k == 0)
      e = poly_pass<-1>(logs[k], LoadPairInt64{a, b, na, nb}, dst, log_len, log_m, batch, st,
                        ftt);
    else
      e = poly_pass<-1>(logs[k], LC{R[(k - 1) % 2], L}, dst, log_len, log_m, batch, st, ftt);
    if (e != cudaSuccess) return e;
    log_m += logs[k];
  }
  double2 *Z = R[(P - 1) % 2];

  // 2 + 3. y = IFFT_{L/2}(Y) with Y formed in the first pass's loads (from Z,
  // which that pass only reads); the last pass rounds into c.  Intermediates
  // alternate between the other buffer and Z's.
  int ilogs[8];
  const int IP = split_passes(log_len - 1, ilogs);
  const LoadCombine comb{Z, tw_lo, tw_hi, lb, L};
  const StoreRoundPairsInt64 round_store{c, nc};
  double2 *bufs[2] = {R[P % 2], Z};
  const double2 *src = nullptr;
  log_m = 0;
  for (int k = 0; k < IP; ++k) {
    const bool last = k == IP - 1;
    double2 *dst = bufs[k % 2];
    if (k == 0) {
      e = last ? poly_pass<+1>(ilogs[k], comb, round_store, log_len - 1, log_m, batch, st, itt)
               : poly_pass<+1>(ilogs[k], comb, SC{dst, H}, log_len - 1, log_m, batch, st, itt);
    } else {
      e = last ? poly_pass<+1>(ilogs[k], LC{src, H}, round_store, log_len - 1, log_m, batch, st,
                               itt)
               : poly_pass<+1>(ilogs[k], LC{src, H}, SC{dst, H}, log_len - 1, log_m, batch, st,
                               itt);
    }
    if (e != cudaSuccess) return e;
    src = dst;
    log_m += ilogs[k];
  }
  return cudaSuccess;
}

int polymul_num_kernels(int log_len) {
  int logs[8];
  return 3 + split_passes(log_len, logs) + split_passes(log_len - 1, logs);
}

}  // namespace fftgb
