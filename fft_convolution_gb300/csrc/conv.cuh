// conv.cuh -- linear convolution of signals through the transform:
// y = x * h, y_k = sum_i x_i h_{k-i} (k < nx + nh - 1), computed as
// IFFT_L( FFT_L(x zero-padded) . FFT_L(h zero-padded) ) with L the smallest
// power of two >= nx + nh - 1 -- the coefficient convolution and the
// "transform, pointwise product, inverse transform" pipeline of "FFT on
// GPU" (polynomial-multiplication section), applied to complex or real
// samples.
//
// * The filter spectra H = FFT_L(h) (one shared filter, or one per row) are
//   computed first into scratch.
// * L <= 2^14 (fp32) / 2^13 (fp64): one kernel per batch does, for each row,
//   load (with the zero padding) -> on-chip forward transform -> product with
//   H -> on-chip inverse transform -> store of the first nx + nh - 1
//   outputs.  Each signal is read from HBM once and its result written once.
// * Longer L: the multi-pass Stockham kernels of fft_pass.cuh, with the
//   padding fused into the first forward pass's loads, the product with H
//   into the last forward pass's stores, and the truncation into the last
//   inverse pass's stores.
// * Real signals with one shared real filter travel in pairs: row 2j as the
//   real part and row 2j+1 as the imaginary part of one complex signal.
//   Because h is real, (x_a + i x_b) * h = x_a * h + i (x_b * h) with both
//   products real, so the result's real and imaginary parts are the two
//   outputs.  Real signals with a filter per row run one row per complex
//   signal (imaginary part zero).
#pragma once

#include "fft_pass.cuh"
#include "fft_rows.cuh"

namespace fftgb {
// Kernels and their launchers have internal linkage (one copy per
// translation unit: conv_f32.cu, conv_f64.cu).
namespace {

enum ConvKind { CONV_COMPLEX = 0, CONV_REAL_PAIRS = 1, CONV_REAL_SINGLE = 2 };

// Sample `idx` of transform row r (complex value), zero beyond n.
template <typename T, int KIND> struct ConvSource {
  const void *p;
  long long n;      // samples per source row
  long long rows;   // source rows (for pairs: the last pair may be half)
  __device__ __forceinline__ vec2_t<T> operator()(long long r, long long idx) const {
    using V = vec2_t<T>;
    if (idx >= n) return make_c<V>((T)0, (T)0);
    if constexpr (KIND == CONV_COMPLEX) {
      return static_cast<const V *>(p)[r * n + idx];
    } else if constexpr (KIND == CONV_REAL_PAIRS) {
      const T *q = static_cast<const T *>(p);
      const long long ra = 2 * r, rb = 2 * r + 1;
      return make_c<V>(q[ra * n + idx], rb < rows ? q[rb * n + idx] : (T)0);
    } else {
      return make_c<V>(static_cast<const T *>(p)[r * n + idx], (T)0);
    }
  }
};

// Output sample `idx` of transform row r, only the first n.
template <typename T, int KIND> struct ConvSink {
  void *p;
  long long n;
  long long rows;
  __device__ __forceinline__ void operator()(long long r, long long idx, vec2_t<T> v) const {
    using V = vec2_t<T>;
    if (idx >= n) return;
    if constexpr (KIND == CONV_COMPLEX) {
      static_cast<V *>(p)[r * n + idx] = v;
    } else if constexpr (KIND == CONV_REAL_PAIRS) {
      T *q = static_cast<T *>(p);
      q[2 * r * n + idx] = v.x;
      if (2 * r + 1 < rows) q[(2 * r + 1) * n + idx] = v.y;
    } else {
      static_cast<T *>(p)[r * n + idx] = v.x;
    }
  }
};

// ---------------------------------------------------------------------------
// On-chip path.  MODE 0: filter spectra H[r] = FFT_L(h_r padded).
// MODE 1: y_r = IFFT_L(FFT_L(x_r padded) . H[r or 0]), first ny outputs.
// ---------------------------------------------------------------------------
// Registers capped for 1024 resident threads per SM (four 256-thread
// blocks) in fp32: the fused kernel does twice the on-chip work of a
// transform per byte of HBM traffic, so it needs the occupancy to hide its
// exchanges.  fp64 values take two registers each: 512 threads (128
// registers), which keeps the 16 values a thread holds out of local memory.
template <typename T, int LOGN> struct ConvRowsBounds {
  static constexpr int THREADS = RowsConfig<T, LOGN>::THREADS;
  static constexpr int RESIDENT = sizeof(T) == 8 ? 512 : 1024;
  static constexpr int MIN_BLOCKS = THREADS >= RESIDENT ? 1 : RESIDENT / THREADS;
};

// Src: (row, idx) -> sample (zero beyond the data); Snk: (row, idx, value).
template <typename T, int LOGN, int MODE, class Src, class Snk>
__global__ void __launch_bounds__(ConvRowsBounds<T, LOGN>::THREADS,
                                  ConvRowsBounds<T, LOGN>::MIN_BLOCKS)
    conv_rows_kernel(Src src, Snk dst, vec2_t<T> *H, int h_per_row, long long trows) {
  using V = vec2_t<T>;
  using P = StagePlan<LOGN>;
  constexpr int F = RowsConfig<T, LOGN>::F;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V *smem = reinterpret_cast<V *>(smem_raw);
  const int t = threadIdx.x % P::TP;
  const int f = threadIdx.x / P::TP;
  const long long r = (long long)blockIdx.x * F + f;
  const bool active = r < trows;
  const SmemView<V> sm{smem + f * P::SMEM_ELEMS, 1};

  V x[P::E];
#pragma unroll
  for (int w = 0; w < P::E; ++w)
    x[w] = active ? src(r, t + w * P::TP) : make_c<V>((T)0, (T)0);
  fft_on_chip<LOGN, -1, false, false>(x, t, sm);  // data came from global memory

  if constexpr (MODE == 0) {
    if (active) {
#pragma unroll
      for (int w = 0; w < P::E; ++w) H[r * P::L + t + w * P::TP] = x[w];
    }
  } else {
    const V *hr = H + (h_per_row ? r : 0) * P::L;
#pragma unroll
    for (int w = 0; w < P::E; ++w)
      x[w] = active ? c_scale(c_mul(x[w], hr[t + w * P::TP]), (T)(1.0 / P::L))
                    : make_c<V>((T)0, (T)0);
    fft_on_chip<LOGN, +1>(x, t, sm);
    if (active) {
#pragma unroll
      for (int w = 0; w < P::E; ++w) dst(r, t + w * P::TP, x[w]);
    }
  }
}

template <typename T, int MODE, class Src, class Snk, int LOGN = 1>
cudaError_t launch_conv_rows(int logn, Src src, Snk dst, vec2_t<T> *H, int h_per_row,
                             long long trows, cudaStream_t st) {
  if constexpr (LOGN > RowsMaxLog<T>::value) {
    return cudaErrorInvalidValue;
  } else {
    if (logn != LOGN)
      return launch_conv_rows<T, MODE, Src, Snk, LOGN + 1>(logn, src, dst, H, h_per_row, trows,
                                                           st);
    using C = RowsConfig<T, LOGN>;
    auto kern = conv_rows_kernel<T, LOGN, MODE, Src, Snk>;
    if (C::SMEM > 48 * 1024) {
      static DeviceOnce attr_set;
      const cudaError_t e = smem_limit_once((const void *)kern, C::SMEM, attr_set);
      if (e != cudaSuccess) return e;
    }
    const long long grid = (trows + C::F - 1) / C::F;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, C::THREADS, C::SMEM, st>>>(src, dst, H, h_per_row, trows);
    return cudaGetLastError();
  }
}

// ---------------------------------------------------------------------------
// Multi-pass path: loads / stores for the pass kernels.
// ---------------------------------------------------------------------------
template <typename T, int KIND> struct PassLoadSource {
  ConvSource<T, KIND> s;
  __device__ __forceinline__ vec2_t<T> operator()(long long b, long long pos) const {
    return s(b, pos);
  }
};
template <typename T> struct PassStoreTimesH {
  vec2_t<T> *out;
  const vec2_t<T> *H;
  long long L;
  int h_per_row;
  __device__ __forceinline__ void operator()(long long b, long long pos, vec2_t<T> v) const {
    out[b * L + pos] = c_mul(v, H[(h_per_row ? b * L : 0) + pos]);
  }
};
template <typename T, int KIND> struct PassStoreSink {
  ConvSink<T, KIND> s;
  __device__ __forceinline__ void operator()(long long b, long long pos, vec2_t<T> v) const {
    s(b, pos, v);
  }
};

template <typename T> constexpr int conv_pass_log() { return sizeof(T) == 4 ? 9 : 11; }

// Factors of a multi-pass convolution transform are never below 5 bits
// (fp32 from 2^15, fp64 from 2^14), so the dispatch starts there.
template <typename T, int DIR, class Load, class Store, int LOGL = 5>
cudaError_t conv_pass(int log_l, Load load, Store store, int log_n, int log_m, long long batch,
                      cudaStream_t st) {
  if constexpr (LOGL > conv_pass_log<T>()) {
    return cudaErrorInvalidValue;
  } else {
    if (log_l == LOGL)
      return launch_pass_t<T, LOGL, DIR>(load, store, log_n, log_m, 1, batch, st);
    return conv_pass<T, DIR, Load, Store, LOGL + 1>(log_l, load, store, log_n, log_m, batch, st);
  }
}

inline int conv_split(int log_len, int limit, int *logs) {
  int P = (log_len + limit - 1) / limit;
  if (P < 2) P = 2;
  for (int k = 0; k < P; ++k) logs[k] = log_len / P + (k < log_len % P ? 1 : 0);
  return P;
}

// Forward multi-pass transform of `rows` padded signals from `load`; the
// last pass hands its output to `last`.  Intermediates alternate between
// bufs[0] and bufs[1].
template <typename T, class Load, class Last>
cudaError_t conv_forward_multi(int log_len, Load load, Last last, vec2_t<T> *const *bufs,
                               long long rows, cudaStream_t st) {
  using V = vec2_t<T>;
  const long long L = 1LL << log_len;
  int logs[8];
  const int P = conv_split(log_len, conv_pass_log<T>(), logs);
  int log_m = 0;
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < P; ++k) {
    const bool first = k == 0, final_pass = k == P - 1;
    StoreComplex<V> mid{bufs[k % 2], L};
    LoadComplex<V> prev{bufs[(k + 1) % 2], L};
    if (first)
      e = conv_pass<T, -1>(logs[k], load, mid, log_len, log_m, rows, st);
    else if (final_pass)
      e = conv_pass<T, -1>(logs[k], prev, last, log_len, log_m, rows, st);
    else
      e = conv_pass<T, -1>(logs[k], prev, mid, log_len, log_m, rows, st);
    if (e != cudaSuccess) return e;
    log_m += logs[k];
  }
  return e;
}

template <typename T, int KIND>
cudaError_t convolve_t(const void *x, long long nx, const void *h, long long nh, void *y,
                       long long batch, int h_per_row, int log_len, void *scratch,
                       cudaStream_t st) {
  using V = vec2_t<T>;
  const long long L = 1LL << log_len;
  const long long ny = nx + nh - 1;
  const long long trows = KIND == CONV_REAL_PAIRS ? (batch + 1) / 2 : batch;
  const long long nfilt = h_per_row ? batch : 1;
  V *H = static_cast<V *>(scratch);
  constexpr int HK = KIND == CONV_COMPLEX ? CONV_COMPLEX : CONV_REAL_SINGLE;  // filter samples
  ConvSource<T, HK> hsrc{h, nh, nfilt};
  ConvSource<T, KIND> xsrc{x, nx, batch};
  ConvSink<T, KIND> ysink{y, ny, batch};
  cudaError_t e;
  if (log_len <= RowsMaxLog<T>::value) {
    e = launch_conv_rows<T, 0>(log_len, hsrc, ConvSink<T, HK>{nullptr, 0, 0}, H, 0, nfilt, st);
    if (e != cudaSuccess) return e;
    return launch_conv_rows<T, 1>(log_len, xsrc, ysink, H, h_per_row, trows, st);
  }
  V *bufs[2] = {H + nfilt * L, H + nfilt * L + trows * L};
  // H = FFT(h padded), written straight into H by the last pass.
  e = conv_forward_multi<T>(log_len, PassLoadSource<T, HK>{hsrc}, StoreComplex<V>{H, L}, bufs,
                            nfilt, st);
  if (e != cudaSuccess) return e;
  // X . H: the product is fused into the last forward pass's stores.
  int logs[8];
  const int P = conv_split(log_len, conv_pass_log<T>(), logs);
  V *prod = bufs[(P - 1) % 2];
  e = conv_forward_multi<T>(log_len, PassLoadSource<T, KIND>{xsrc},
                            PassStoreTimesH<T>{prod, H, L, h_per_row}, bufs, trows, st);
  if (e != cudaSuccess) return e;
  // Inverse passes; the last one stores the first ny outputs.
  int log_m = 0;
  const V *src = prod;
  V *alt[2] = {bufs[P % 2], prod};
  for (int k = 0; k < P; ++k) {
    if (k == P - 1) {
      e = conv_pass<T, +1>(logs[k], LoadComplex<V>{src, L}, PassStoreSink<T, KIND>{ysink},
                           log_len, log_m, trows, st);
    } else {
      V *d = alt[k % 2];
      e = conv_pass<T, +1>(logs[k], LoadComplex<V>{src, L}, StoreComplex<V>{d, L}, log_len,
                           log_m, trows, st);
      src = d;
    }
    if (e != cudaSuccess) return e;
    log_m += logs[k];
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace fftgb
