// anylen.cuh -- transforms of any length N (not a power of two).
//
// "FFT on GPU" (section FFT on GPU, and section Algorithm per signal
// Length) falls back to the direct O(N^2) DFT when N is not a power of two
// and names Bluestein's algorithm as the way to any length through a
// power-of-two transform.  Both are here:
//
// * N <= 64: direct DFT, X_k = sum_n x_n W_N^{nk}, one thread per output,
//   the N twiddles and the rows staged in shared memory (dft_small_kernel).
// * N > 64: Bluestein.  With w_n = e^{DIR i pi n^2 / N} (the exponent n^2
//   reduced mod 2N in integers) and nk = (n^2 + k^2 - (k-n)^2) / 2,
//       X_k = w_k sum_n (x_n w_n) conj(w_{k-n}),
//   a linear convolution of a_n = x_n w_n with b_m = conj(w_|m|), done as a
//   cyclic one of power-of-two length M >= 2N - 1 by the convolution
//   kernels of conv.cuh: a_n is formed in the first load, the product with
//   the precomputed B = FFT_M(b) and the final w_k (and 1/N for the
//   inverse) in the stores.
#pragma once

#include "conv.cuh"

namespace fftgb {
namespace {

template <typename T> struct ChirpSource {  // a_n = x_n w_n (n < N), 0 beyond
  const vec2_t<T> *x;
  const vec2_t<T> *w;
  long long N;
  __device__ __forceinline__ vec2_t<T> operator()(long long r, long long idx) const {
    using V = vec2_t<T>;
    return idx < N ? c_mul(x[r * N + idx], w[idx]) : make_c<V>((T)0, (T)0);
  }
};

template <typename T> struct ChirpSink {  // X_k = w_k c_k * scale (k < N)
  vec2_t<T> *y;
  const vec2_t<T> *w;
  long long N;
  T scale;
  __device__ __forceinline__ void operator()(long long r, long long idx, vec2_t<T> v) const {
    if (idx < N) y[r * N + idx] = c_scale(c_mul(v, w[idx]), scale);
  }
};

// b_m = conj(w_m) for 0 <= m < N and b_{M-m} = conj(w_m) for 0 < m < N
// (the negative lags of the linear convolution, wrapped), 0 elsewhere.
template <typename T> struct ChirpFilterSource {
  const vec2_t<T> *w;
  long long N, M;
  __device__ __forceinline__ vec2_t<T> operator()(long long, long long idx) const {
    using V = vec2_t<T>;
    long long m = -1;
    if (idx < N) m = idx;
    else if (idx > M - N) m = M - idx;
    if (m < 0) return make_c<V>((T)0, (T)0);
    const V v = w[m];
    return make_c<V>(v.x, -v.y);
  }
};

template <class Src> struct PassLoadFrom {
  Src s;
  __device__ __forceinline__ auto operator()(long long b, long long pos) const { return s(b, pos); }
};
template <class Snk> struct PassStoreTo {
  Snk s;
  template <typename V>
  __device__ __forceinline__ void operator()(long long b, long long pos, V v) const {
    s(b, pos, v);
  }
};

// w_n = e^{dir i pi (n^2 mod 2N) / N}, computed in fp64 and rounded to T.
template <typename T>
__global__ void chirp_kernel(vec2_t<T> *w, long long N, int dir) {
  const long long n = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const long long e = (long long)(((unsigned long long)n * (unsigned long long)n) %
                                  (unsigned long long)(2 * N));
  double s, c;
  sincospi((double)e / (double)N, &s, &c);
  w[n] = make_c<vec2_t<T>>((T)c, (T)(dir * s));
}

// Direct DFT for N <= 64: a block holds 256 / N rows (whole rows) and the N
// twiddles W^m = e^{dir 2 pi i m / N} (fp64 sincospi, rounded to T); thread
// (row, k) sums x_n W^{(n k) mod N} over n in order.
template <typename T>
__global__ void dft_small_kernel(const vec2_t<T> *x, vec2_t<T> *y, int N, long long rows,
                                 int dir, T scale) {
  using V = vec2_t<T>;
  __shared__ V tw[64];
  __shared__ V xs[256];
  const int per = 256 / N;
  const int rr = threadIdx.x / N, k = threadIdx.x % N;
  const long long r = (long long)blockIdx.x * per + rr;
  const bool active = rr < per && r < rows;
  if (threadIdx.x < N) {
    double s, c;
    sincospi(2.0 * (double)threadIdx.x / (double)N, &s, &c);
    tw[threadIdx.x] = make_c<V>((T)c, (T)(dir * s));
  }
  if (active) xs[rr * N + k] = x[r * N + k];
  __syncthreads();
  if (!active) return;
  V acc = make_c<V>((T)0, (T)0);
  int m = 0;  // (n k) mod N, stepped by k
  for (int n = 0; n < N; ++n) {
    acc = c_add(acc, c_mul(xs[rr * N + n], tw[m]));
    m += k;
    if (m >= N) m -= N;
  }
  y[r * N + k] = c_scale(acc, scale);
}

// The precomputed state of a Bluestein plan.
template <typename T> struct BluesteinState {
  vec2_t<T> *w;   // N chirp values for the plan's direction
  vec2_t<T> *B;   // FFT_M(b), M values
  vec2_t<T> *ws;  // multi-pass work: 2 * batch * M values (M beyond on-chip)
};

// B = FFT_M(b) (on stream st).
template <typename T>
cudaError_t bluestein_prepare_t(long long N, int log_m, int dir, BluesteinState<T> s,
                                cudaStream_t st) {
  using V = vec2_t<T>;
  const long long M = 1LL << log_m;
  chirp_kernel<T><<<(unsigned)((N + 255) / 256), 256, 0, st>>>(s.w, N, dir);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ChirpFilterSource<T> bsrc{s.w, N, M};
  if (log_m <= RowsMaxLog<T>::value)
    return launch_conv_rows<T, 0>(log_m, bsrc, ChirpSink<T>{nullptr, nullptr, 0, (T)0}, s.B, 0, 1,
                                  st);
  V *bufs[2] = {s.ws, s.ws + M};
  return conv_forward_multi<T>(log_m, PassLoadFrom<ChirpFilterSource<T>>{bsrc},
                               StoreComplex<V>{s.B, M}, bufs, 1, st);
}

template <typename T>
cudaError_t bluestein_exec_t(const void *in, void *out, long long N, long long batch, int log_m,
                             T scale, BluesteinState<T> s, cudaStream_t st) {
  using V = vec2_t<T>;
  const long long M = 1LL << log_m;
  ChirpSource<T> src{static_cast<const V *>(in), s.w, N};
  ChirpSink<T> snk{static_cast<V *>(out), s.w, N, scale};
  if (log_m <= RowsMaxLog<T>::value)
    return launch_conv_rows<T, 1>(log_m, src, snk, s.B, 0, batch, st);
  V *bufs[2] = {s.ws, s.ws + batch * M};
  int logs[8];
  const int P = conv_split(log_m, conv_pass_log<T>(), logs);
  V *prod = bufs[(P - 1) % 2];
  cudaError_t e = conv_forward_multi<T>(log_m, PassLoadFrom<ChirpSource<T>>{src},
                                        PassStoreTimesH<T>{prod, s.B, M, 0}, bufs, batch, st);
  if (e != cudaSuccess) return e;
  int log_acc = 0;
  const V *cur = prod;
  V *alt[2] = {bufs[P % 2], prod};
  for (int k = 0; k < P; ++k) {
    if (k == P - 1) {
      e = conv_pass<T, +1>(logs[k], LoadComplex<V>{cur, M}, PassStoreTo<ChirpSink<T>>{snk}, log_m,
                           log_acc, batch, st);
    } else {
      V *d = alt[k % 2];
      e = conv_pass<T, +1>(logs[k], LoadComplex<V>{cur, M}, StoreComplex<V>{d, M}, log_m, log_acc,
                           batch, st);
      cur = d;
    }
    if (e != cudaSuccess) return e;
    log_acc += logs[k];
  }
  return cudaSuccess;
}

template <typename T>
cudaError_t dft_small_t(const void *in, void *out, int N, long long batch, int dir, T scale,
                        cudaStream_t st) {
  using V = vec2_t<T>;
  const int per = 256 / N;
  const long long grid = (batch + per - 1) / per;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dft_small_kernel<T><<<(unsigned)grid, 256, 0, st>>>(static_cast<const V *>(in),
                                                      static_cast<V *>(out), N, batch, dir, scale);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fftgb
