// real.cuh -- transforms of real sequences (half spectrum in, or out).
//
// For real x the DFT of "FFT on GPU" (section Discrete Fourier Transform)
// has X_{N-k} = conj(X_k), so bins 0 .. N/2 carry all of it.  For even
// N = 2H the real row is read as H complex values z_n = x_{2n} + i x_{2n+1}
// (the same bytes) and transformed at half length; with Z = FFT_H(z) and
// E_k, O_k the transforms of the even and odd samples (the page's even/odd
// split, section Fast Fourier Transform):
//   E_k = (Z_k + conj(Z_{H-k})) / 2,    O_k = -i (Z_k - conj(Z_{H-k})) / 2,
//   X_k = E_k + W_N^k O_k,              X_{H-k} = conj(E_k - W_N^k O_k)
// (indices of Z mod H; k = 0 gives X_0 and X_H).  The inverse runs the same
// relations backwards:
//   E_k = (X_k + conj(X_{H-k})) / 2,    O_k = W_N^{-k} (X_k - conj(X_{H-k})) / 2,
//   Z_k = E_k + i O_k,  Z_{H-k} = conj(E_k) + i conj(O_k),
// and x_{2n} + i x_{2n+1} = (1/H) sum_k Z_k W_H^{-nk}.  The imaginary parts of
// X_0 and X_H are dropped first (they only add imaginary terms to x).
//
// * H <= 2^14 (fp32) / 2^13 (fp64), power of two: one kernel per direction,
//   the half-length transform on chip and the mirror pairs (k, H-k)
//   exchanged through shared memory (r2c_rows_kernel, c2r_rows_kernel).
// * Otherwise: a complex plan of length H between a pre or post kernel that
//   applies the relations above over HBM (real_post_kernel,
//   real_pre_kernel); odd N goes through a complex plan of length N with the
//   samples widened to complex (imaginary part 0) and the spectrum extended
//   by X_{N-k} = conj(X_k).
#pragma once

#include "fft_rows.cuh"

namespace fftgb {
namespace {

template <typename T, int LOGH> struct RealRowsConfig {
  using P = StagePlan<LOGH>;
  static constexpr int F = RowsConfig<T, LOGH>::F;
  static constexpr int THREADS = RowsConfig<T, LOGH>::THREADS;
  // The exchanges of the transform, and the mirror exchange (H + 1 values).
  static constexpr int ELEMS = P::L + P::L / 16 + 1;
  static constexpr size_t SMEM = (size_t)F * ELEMS * sizeof(vec2_t<T>);
};

template <typename V> __device__ __forceinline__ V c_conj(V a) {
  a.y = -a.y;
  return a;
}

// Calls f(w, a s^w) for w = 0 .. E-1 in increasing w, the factors built as
// a, a s, a s^2, a s^3 and then stepped by s^4 (at most five products deep,
// as apply_geometric), so that a caller can finish element w before the
// next factor is formed and keep only the elements themselves live.
template <int E, typename V, class Fn>
__device__ __forceinline__ void geometric_each(V a, V s, Fn f) {
  if constexpr (E >= 4 && E % 4 == 0) {
    const V s2 = c_mul(s, s), s4 = c_mul(s2, s2);
    V q[4];
    q[0] = a;
    q[1] = c_mul(a, s);
    q[2] = c_mul(a, s2);
    q[3] = c_mul(q[1], s2);
#pragma unroll
    for (int blk = 0; blk < E / 4; ++blk) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f(4 * blk + j, q[j]);
        if (blk + 1 < E / 4) q[j] = c_mul(q[j], s4);
      }
    }
  } else {
    V pw[E];
    powers<E>(s, pw);
#pragma unroll
    for (int w = 0; w < E; ++w) f(w, c_mul(a, pw[w]));
  }
}

template <typename T, int LOGH> struct RealRowsBounds {
  // Four blocks of 256 threads per SM in fp32 (64 registers a thread); two
  // in fp64 (128 registers: the values a thread holds take two each).
  static constexpr int RESIDENT = sizeof(T) == 8 ? 512 : 1024;
  static constexpr int MIN_BLOCKS = RealRowsConfig<T, LOGH>::THREADS >= RESIDENT
                                        ? 1
                                        : RESIDENT / RealRowsConfig<T, LOGH>::THREADS;
};

// Forward: batch rows of N = 2H reals (read as H complex) -> batch rows of
// H + 1 complex bins.
template <typename T, int LOGH>
__global__ void __launch_bounds__(RealRowsConfig<T, LOGH>::THREADS, RealRowsBounds<T, LOGH>::MIN_BLOCKS)
    r2c_rows_kernel(const vec2_t<T> *in, vec2_t<T> *out, long long batch) {
  using V = vec2_t<T>;
  using P = StagePlan<LOGH>;
  using C = RealRowsConfig<T, LOGH>;
  constexpr int H = P::L;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V *smem = reinterpret_cast<V *>(smem_raw);

  const int t = threadIdx.x % P::TP;
  const int f = threadIdx.x / P::TP;
  const long long r = (long long)blockIdx.x * C::F + f;
  const bool active = r < batch;

  // Programmatic dependent launch, as the row kernel: wait for the
  // previous kernel before reading, let the next one be scheduled once
  // this block holds its data.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  V x[P::E];
  if (active) {
    const V *src = in + r * H;
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = src[t + w * P::TP];
  } else {
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = make_c<V>((T)0, (T)0);
  }
  asm volatile("griddepcontrol.launch_dependents;");
  const SmemView<V> sm{smem + f * C::ELEMS, 1};
  fft_on_chip<LOGH, -1, false, false>(x, t, sm);  // data came from global memory

  // x[w] = Z_k, k = t + w TP.  Mirror through shared memory.
  __syncthreads();
#pragma unroll
  for (int w = 0; w < P::E; ++w) sm.st(t + w * P::TP, x[w]);
  __syncthreads();
  // X_k = E_k + W_N^k O_k with W_N^k = W_N^t (W_N^TP)^w, N = 2H; x[w]
  // becomes X_k.  X_H = E_0 - O_0 is kept aside by thread 0.
  V xh = make_c<V>((T)0, (T)0);
  geometric_each<P::E>(twiddle<-1>((long long)t, LOGH + 1, T()),
                       twiddle<-1>((long long)P::TP, LOGH + 1, T()), [&](int w, V wk) {
                         const int k = t + w * P::TP;
                         const V zm = c_conj(sm.ld((H - k) & (H - 1)));
                         const V s = c_add(x[w], zm), d = c_sub(x[w], zm);
                         const V e = make_c<V>((T)0.5 * s.x, (T)0.5 * s.y);
                         const V o = c_mul(make_c<V>((T)0.5 * d.y, (T)-0.5 * d.x), wk);  // -i d/2
                         if (w == 0) xh = c_sub(e, o);
                         x[w] = c_add(e, o);
                       });
  if (active) {
    V *dst = out + r * (H + 1);
#pragma unroll
    for (int w = 0; w < P::E; ++w) dst[t + w * P::TP] = x[w];
    if (t == 0) dst[H] = xh;
  }
}

// Inverse: batch rows of H + 1 complex bins -> batch rows of N = 2H reals
// (written as H complex), scaled by 1/N.
template <typename T, int LOGH>
__global__ void __launch_bounds__(RealRowsConfig<T, LOGH>::THREADS, RealRowsBounds<T, LOGH>::MIN_BLOCKS)
    c2r_rows_kernel(const vec2_t<T> *in, vec2_t<T> *out, long long batch) {
  using V = vec2_t<T>;
  using P = StagePlan<LOGH>;
  using C = RealRowsConfig<T, LOGH>;
  constexpr int H = P::L;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V *smem = reinterpret_cast<V *>(smem_raw);

  const int t = threadIdx.x % P::TP;
  const int f = threadIdx.x / P::TP;
  const long long r = (long long)blockIdx.x * C::F + f;
  const bool active = r < batch;
  const SmemView<V> sm{smem + f * C::ELEMS, 1};

  asm volatile("griddepcontrol.wait;" ::: "memory");  // as in r2c_rows_kernel
  V x[P::E];
  if (active) {
    const V *src = in + r * (H + 1);
#pragma unroll
    for (int w = 0; w < P::E; ++w) {
      V v = src[t + w * P::TP];
      if (t == 0 && w == 0) v.y = (T)0;  // Im X_0 dropped
      x[w] = v;
      sm.st(t + w * P::TP, v);
    }
    if (t == 0) {
      V v = src[H];
      v.y = (T)0;  // Im X_H dropped
      sm.st(H, v);
    }
  } else {
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = make_c<V>((T)0, (T)0);
  }
  asm volatile("griddepcontrol.launch_dependents;");
  __syncthreads();
  // Z_k = 2E_k + i (2 O_k), 2 O_k = W_N^{-k} (X_k - conj(X_{H-k})) (the
  // factor 1/2 joins 1/H at the store).
  geometric_each<P::E>(twiddle<1>((long long)t, LOGH + 1, T()),
                       twiddle<1>((long long)P::TP, LOGH + 1, T()), [&](int w, V wk) {
                         const int k = t + w * P::TP;
                         const V xm = active ? c_conj(sm.ld(H - k)) : make_c<V>((T)0, (T)0);
                         const V d = c_mul(c_sub(x[w], xm), wk);
                         const V e2 = c_add(x[w], xm);
                         x[w] = make_c<V>(e2.x - d.y, e2.y + d.x);
                       });
  // The transform's first exchange waits for every thread's mirror reads.
  fft_on_chip<LOGH, 1>(x, t, sm);
  if (active) {
    V *dst = out + r * H;
    const T scale = (T)(0.5 / H);
#pragma unroll
    for (int w = 0; w < P::E; ++w) dst[t + w * P::TP] = c_scale(x[w], scale);
  }
}

template <typename T, int LOGH, bool FWD>
cudaError_t launch_real_rows_t(const void *in, void *out, long long batch, cudaStream_t st) {
  using C = RealRowsConfig<T, LOGH>;
  using V = vec2_t<T>;
  auto kern = FWD ? r2c_rows_kernel<T, LOGH> : c2r_rows_kernel<T, LOGH>;
  if (C::SMEM > 48 * 1024) {
    static DeviceOnce attr_set;
    const cudaError_t e = smem_limit_once((const void *)kern, C::SMEM, attr_set);
    if (e != cudaSuccess) return e;
  }
  const long long grid = (batch + C::F - 1) / C::F;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const V *>(in), static_cast<V *>(out), batch);
}

template <typename T, bool FWD, int LOGH = 0>
cudaError_t dispatch_real_rows(int logh, const void *in, void *out, long long batch,
                               cudaStream_t st) {
  if constexpr (LOGH > RowsMaxLog<T>::value) {
    return cudaErrorInvalidValue;
  } else {
    if (logh == LOGH) return launch_real_rows_t<T, LOGH, FWD>(in, out, batch, st);
    return dispatch_real_rows<T, FWD, LOGH + 1>(logh, in, out, batch, st);
  }
}

// ---------------------------------------------------------------------------
// Over HBM, around a complex plan.
// ---------------------------------------------------------------------------

// W_N^e for 0 <= e < N from two tables: lo[j] = W_N^j (j < S = 2^log_s),
// hi[i] = W_N^{i S}; W_N^e = hi[e >> log_s] lo[e & (S - 1)].
template <typename V> struct SplitTwiddle {
  const V *lo, *hi;
  int log_s;
  __device__ __forceinline__ V operator()(long long e) const {
    return c_mul(hi[e >> log_s], lo[e & ((1LL << log_s) - 1)]);
  }
};

// Both tables of the forward root W_N = e^{-2 pi i / N}: lo has S entries,
// hi has nhi; each from an fp64 sincospi of the exponent reduced mod N in
// integers, rounded once to T.
template <typename T>
__global__ void real_twiddle_kernel(vec2_t<T> *lo, vec2_t<T> *hi, long long n, int log_s,
                                    long long nhi) {
  const long long S = 1LL << log_s;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  long long e;
  vec2_t<T> *dst;
  if (i < S) {
    e = i % n;
    dst = lo + i;
  } else if (i < S + nhi) {
    e = (long long)(((unsigned long long)(i - S) * (unsigned long long)S) % (unsigned long long)n);
    dst = hi + (i - S);
  } else {
    return;
  }
  double s, c;
  sincospi(2.0 * (double)e / (double)n, &s, &c);
  *dst = make_c<vec2_t<T>>((T)c, (T)-s);
}

inline unsigned aux_grid(long long items) {
  long long g = (items + 255) / 256;
  const long long cap = 152LL * 16;
  if (g > cap) g = cap;
  return (unsigned)(g < 1 ? 1 : g);
}

// Forward post-processing: Z (batch x H) -> X (batch x (H + 1)); one item per
// mirror pair (k, H - k), k = 0 .. H/2.
template <typename T>
__global__ void real_post_kernel(const vec2_t<T> *Z, vec2_t<T> *X, long long H, long long batch,
                                 SplitTwiddle<vec2_t<T>> W) {
  using V = vec2_t<T>;
  const long long per = H / 2 + 1, total = per * batch;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long r = it / per, k = it - r * per;
    const V *z = Z + r * H;
    V *x = X + r * (H + 1);
    const V zk = z[k], zm = c_conj(z[k == 0 ? 0 : H - k]);
    const V s = c_add(zk, zm), d = c_sub(zk, zm);
    const V e = make_c<V>((T)0.5 * s.x, (T)0.5 * s.y);
    const V o = c_mul(make_c<V>((T)0.5 * d.y, (T)-0.5 * d.x), W(k));
    x[k] = c_add(e, o);
    if (H - k != k) x[H - k] = c_conj(c_sub(e, o));
  }
}

// Inverse pre-processing: X (batch x (H + 1)) -> Z (batch x H), for a
// complex inverse of length H (with its 1/H) to finish.
template <typename T>
__global__ void real_pre_kernel(const vec2_t<T> *X, vec2_t<T> *Z, long long H, long long batch,
                                SplitTwiddle<vec2_t<T>> W) {
  using V = vec2_t<T>;
  const long long per = H / 2 + 1, total = per * batch;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long r = it / per, k = it - r * per;
    const V *x = X + r * (H + 1);
    V *z = Z + r * H;
    V xk = x[k], xm = x[H - k];
    if (k == 0) {
      xk.y = (T)0;
      xm.y = (T)0;
    }
    xm = c_conj(xm);
    const V s = c_add(xk, xm), d = c_sub(xk, xm);
    const V e = make_c<V>((T)0.5 * s.x, (T)0.5 * s.y);
    const V o = c_mul(make_c<V>((T)0.5 * d.x, (T)0.5 * d.y), c_conj(W(k)));
    z[k] = make_c<V>(e.x - o.y, e.y + o.x);  // E + i O
    if (k != 0 && H - k != k) z[H - k] = make_c<V>(e.x + o.y, -e.y + o.x);  // conj(E) + i conj(O)
  }
}

// Odd N: real samples widened to complex (imaginary part 0).
template <typename T>
__global__ void real_widen_kernel(const T *x, vec2_t<T> *z, long long count) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (long long)gridDim.x * blockDim.x)
    z[i] = make_c<vec2_t<T>>(x[i], (T)0);
}

// Odd N: the first N/2 + 1 bins of each transformed row.
template <typename T>
__global__ void real_narrow_kernel(const vec2_t<T> *z, vec2_t<T> *X, long long n, long long batch) {
  const long long per = n / 2 + 1, total = per * batch;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long r = it / per, k = it - r * per;
    X[it] = z[r * n + k];
  }
}

// Odd N: the full spectrum Y_k = X_k (k <= N/2), conj(X_{N-k}) (k > N/2),
// with Im X_0 dropped.
template <typename T>
__global__ void real_extend_kernel(const vec2_t<T> *X, vec2_t<T> *z, long long n, long long batch) {
  using V = vec2_t<T>;
  const long long per = n / 2 + 1, total = n * batch;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long r = it / n, k = it - r * n;
    const V *x = X + r * per;
    V v = 2 * k <= n ? x[k] : c_conj(x[n - k]);
    if (k == 0) v.y = (T)0;
    z[it] = v;
  }
}

// Odd N: real parts of the inverse-transformed rows.
template <typename T>
__global__ void real_part_kernel(const vec2_t<T> *z, T *x, long long count) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (long long)gridDim.x * blockDim.x)
    x[i] = z[i].x;
}

template <typename T>
cudaError_t real_aux_t(int op, const RealAuxArgs &a, cudaStream_t st) {
  using V = vec2_t<T>;
  const long long n = a.len;
  const V *lo = static_cast<const V *>(a.lo), *hi = static_cast<const V *>(a.hi);
  const SplitTwiddle<V> W{lo, hi, a.log_s};
  switch (op) {
    case REAL_TABLES: {
      const long long items = (1LL << a.log_s) + a.nhi;
      real_twiddle_kernel<T><<<(unsigned)((items + 255) / 256), 256, 0, st>>>(
          static_cast<V *>(const_cast<void *>(a.lo)), static_cast<V *>(const_cast<void *>(a.hi)),
          n, a.log_s, a.nhi);
      break;
    }
    case REAL_POST:
      real_post_kernel<T><<<aux_grid((n / 2 + 1) * a.batch), 256, 0, st>>>(
          static_cast<const V *>(a.in), static_cast<V *>(a.out), n, a.batch, W);
      break;
    case REAL_PRE:
      real_pre_kernel<T><<<aux_grid((n / 2 + 1) * a.batch), 256, 0, st>>>(
          static_cast<const V *>(a.in), static_cast<V *>(a.out), n, a.batch, W);
      break;
    case REAL_WIDEN:
      real_widen_kernel<T><<<aux_grid(n * a.batch), 256, 0, st>>>(
          static_cast<const T *>(a.in), static_cast<V *>(a.out), n * a.batch);
      break;
    case REAL_NARROW:
      real_narrow_kernel<T><<<aux_grid((n / 2 + 1) * a.batch), 256, 0, st>>>(
          static_cast<const V *>(a.in), static_cast<V *>(a.out), n, a.batch);
      break;
    case REAL_EXTEND:
      real_extend_kernel<T><<<aux_grid(n * a.batch), 256, 0, st>>>(
          static_cast<const V *>(a.in), static_cast<V *>(a.out), n, a.batch);
      break;
    case REAL_PART:
      real_part_kernel<T><<<aux_grid(n * a.batch), 256, 0, st>>>(
          static_cast<const V *>(a.in), static_cast<T *>(a.out), n * a.batch);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace
}  // namespace fftgb
