// fft_device.cuh -- register-level butterflies, twiddles and the on-chip
// Stockham engine shared by every transform kernel of the library.
//
// Definitions followed:
//  * DFT and roots of unity: X_k = sum_n x_n omega_N^{kn},
//    omega_N = e^{-i 2 pi / N} ("FFT on GPU", sections Discrete Fourier
//    Transform and Primitive Root of Unity); inverse kernels use the
//    conjugate root.
//  * Butterfly a +- w b ("The Butterfly: One Thread, One Output", gpu.rocks;
//    "FFT on GPU", section Fast Fourier Transform).  Small DFTs held in
//    registers are built from these butterflies by the even/odd split of
//    the same section.
//  * Stockham autosort stage ("Stockham FFT Butterfly Algorithm in Parallel
//    GLSL", section Execution via GLSL Compute Shaders, items 2-3), here in
//    its radix-R form: a stage with previous block length m and radix R
//    computes, for every butterfly index i = q*m + p (p < m) and v < R,
//        out[q*R*m + p + v*m] = sum_{u<R} W_R^{uv} W_{Rm}^{p*u} in[i + u*N/R]
//    which for R = 2 is exactly the page's stage (j = i, k = j + N/2,
//    r = (x mod 2m) * N/(2m)).  Input and output are in natural order; no
//    bit-reversal permutation is ever applied.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fftgb {

template <typename T> struct Vec2;
template <> struct Vec2<float> { using type = float2; };
template <> struct Vec2<double> { using type = double2; };
template <typename T> using vec2_t = typename Vec2<T>::type;

template <typename V> __device__ __forceinline__ V make_c(decltype(V::x) re, decltype(V::x) im) {
  V r;
  r.x = re;
  r.y = im;
  return r;
}
template <typename V> __device__ __forceinline__ V c_add(V a, V b) {
  return make_c<V>(a.x + b.x, a.y + b.y);
}
template <typename V> __device__ __forceinline__ V c_sub(V a, V b) {
  return make_c<V>(a.x - b.x, a.y - b.y);
}
template <typename V> __device__ __forceinline__ V c_mul(V a, V b) {
  return make_c<V>(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
template <typename V> __device__ __forceinline__ V c_scale(V a, decltype(V::x) s) {
  return make_c<V>(a.x * s, a.y * s);
}
// Multiply by DIR*i (DIR = -1: by -i; DIR = +1: by +i).
template <int DIR, typename V> __device__ __forceinline__ V c_mul_diri(V a) {
  if constexpr (DIR < 0) return make_c<V>(a.y, -a.x);
  else return make_c<V>(-a.y, a.x);
}

// cos(2 pi j / 16) for j in [0, 16): the only constants a radix <= 16
// butterfly needs.
__host__ __device__ constexpr double cos16(int j) {
  return j == 0    ? 1.0
         : j == 1  ? 0.923879532511286756128183189396788933
         : j == 2  ? 0.707106781186547524400844362104849039
         : j == 3  ? 0.382683432365089771728459984030398866
         : j == 4  ? 0.0
         : j == 5  ? -0.382683432365089771728459984030398866
         : j == 6  ? -0.707106781186547524400844362104849039
         : j == 7  ? -0.923879532511286756128183189396788933
         : j == 8  ? -1.0
         : j == 9  ? -0.923879532511286756128183189396788933
         : j == 10 ? -0.707106781186547524400844362104849039
         : j == 11 ? -0.382683432365089771728459984030398866
         : j == 12 ? 0.0
         : j == 13 ? 0.382683432365089771728459984030398866
         : j == 14 ? 0.707106781186547524400844362104849039
                   : 0.923879532511286756128183189396788933;
}

// a * W_R^K with W_R = e^{DIR i 2 pi / R}, R | 16, K a compile-time constant.
template <int R, int K, int DIR, typename V> __device__ __forceinline__ V tw_const(V a) {
  using T = decltype(V::x);
  constexpr int j = ((K % R) * (16 / R)) & 15;
  if constexpr (j == 0) {
    return a;
  } else if constexpr (j == 4) {
    return c_mul_diri<DIR>(a);
  } else if constexpr (j == 8) {
    return make_c<V>(-a.x, -a.y);
  } else if constexpr (j == 12) {
    return c_mul_diri<-DIR>(a);
  } else {
    constexpr T c = (T)cos16(j);
    constexpr T s = (T)(DIR * cos16((j + 12) & 15));  // DIR * sin(2 pi j / 16)
    return c_mul(a, make_c<V>(c, s));
  }
}

// Combine step of the even/odd split: x[k] = e[k] + W_R^k o[k],
// x[k + R/2] = e[k] - W_R^k o[k].
template <int R, int DIR, int K, typename V>
__device__ __forceinline__ void combine(V *x, const V *e, const V *o) {
  if constexpr (K < R / 2) {
    V t = tw_const<R, K, DIR>(o[K]);
    x[K] = c_add(e[K], t);
    x[K + R / 2] = c_sub(e[K], t);
    combine<R, DIR, K + 1>(x, e, o);
  }
}

// In-register DFT of length R (1, 2, 4, 8, 16), natural order in and out.
template <int R, int DIR, typename V> __device__ __forceinline__ void dft_reg(V *x) {
  if constexpr (R == 2) {
    V a = x[0], b = x[1];
    x[0] = c_add(a, b);
    x[1] = c_sub(a, b);
  } else if constexpr (R > 2) {
    V e[R / 2], o[R / 2];
#pragma unroll
    for (int k = 0; k < R / 2; ++k) {
      e[k] = x[2 * k];
      o[k] = x[2 * k + 1];
    }
    dft_reg<R / 2, DIR>(e);
    dft_reg<R / 2, DIR>(o);
    combine<R, DIR, 0>(x, e, o);
  }
}

// ---------------------------------------------------------------------------
// Twiddles computed on the fly (no lookup table; the GLSL page's choice of
// trading a little ALU work for memory bandwidth).
// ---------------------------------------------------------------------------

// W_M^e = e^{DIR i 2 pi e / M} for M = 2^log2m, the integer exponent first
// reduced mod M.  Arguments of sincospi are formed exactly (integer times a
// power of two), so the only rounding is sincospi's own.
template <int DIR> __device__ __forceinline__ float2 twiddle(long long e, int log2m, float) {
  const long long mask = (1LL << log2m) - 1;
  e &= mask;
  float s, c;
  if (log2m <= 24) {
    sincospif(ldexpf((float)e, 1 - log2m), &s, &c);
    return make_c<float2>(c, DIR * s);
  }
  // Exponent wider than the float mantissa: W^e = W^{hi * 2^12} W^{lo}.
  const long long lo = e & 4095, hi = e >> 12;
  float s1, c1;
  sincospif(ldexpf((float)hi, 13 - log2m), &s, &c);
  sincospif(ldexpf((float)lo, 1 - log2m), &s1, &c1);
  return c_mul(make_c<float2>(c, DIR * s), make_c<float2>(c1, DIR * s1));
}
template <int DIR> __device__ __forceinline__ double2 twiddle(long long e, int log2m, double) {
  const long long mask = (1LL << log2m) - 1;
  e &= mask;
  double s, c;
  sincospi(ldexp((double)e, 1 - log2m), &s, &c);
  return make_c<double2>(c, DIR * s);
}

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v >> 1); }
__host__ __device__ constexpr int high_bit(int v) { return 1 << ilog2(v); }

// p[u] = w^u for u in [0, R): powers by squaring / one product each
// (p[2^a] = p[2^(a-1)]^2, p[2^a + b] = p[2^a] p[b]), so no power is more
// than log2(R) multiplications deep.
template <int U, int R, typename V> __device__ __forceinline__ void powers_from(V *p) {
  if constexpr (U < R) {
    constexpr int hb = high_bit(U);
    if constexpr (U == hb) p[U] = c_mul(p[U / 2], p[U / 2]);
    else p[U] = c_mul(p[hb], p[U - hb]);
    powers_from<U + 1, R>(p);
  }
}
template <int R, typename V> __device__ __forceinline__ void powers(V w, V *p) {
  using T = decltype(V::x);
  p[0] = make_c<V>((T)1, (T)0);
  if constexpr (R > 1) p[1] = w;
  powers_from<2, R>(p);
}

// ---------------------------------------------------------------------------
// Stage plan of an on-chip transform of length L = 2^LOGL.
//   E  = elements each thread holds (16, or L if L < 16)
//   TP = threads per transform (L / E)
//   stage 0 has radix R0 = 2^(LOGL - 4*(NS-1)) in {2,4,8,16}, later stages
//   radix 16; stage k > 0 starts from blocks of length m_k = R0 * 16^(k-1).
// ---------------------------------------------------------------------------
template <int LOGL> struct StagePlan {
  static constexpr int L = 1 << LOGL;
  static constexpr int E = L < 16 ? L : 16;
  static constexpr int TP = L / E;
  static constexpr int NS = LOGL == 0 ? 0 : (LOGL + 3) / 4;
  static constexpr int R0 = NS == 0 ? 1 : 1 << (LOGL - 4 * (NS - 1));
  __host__ __device__ static constexpr int radix(int k) { return k == 0 ? R0 : 16; }
  __host__ __device__ static constexpr int log_m(int k) {
    return k == 0 ? 0 : (LOGL - 4 * (NS - 1)) + 4 * (k - 1);
  }
  // Shared-memory elements needed for the exchanges (padded by one per 16).
  static constexpr int SMEM_ELEMS = NS > 1 ? L + L / 16 : 0;
  // Twiddle table (optional): stage k > 0 keeps W_{R m}^{p u} for u < R,
  // p < m at tw_offset(k) + u*m + p.
  __host__ __device__ static constexpr int tw_offset(int k) {
    return k <= 1 ? 0 : tw_offset(k - 1) + (radix(k - 1) << log_m(k - 1));
  }
  static constexpr int TW_ELEMS = NS > 1 ? tw_offset(NS) : 0;
};

// Padded shared-memory position: one spare slot every 16 elements keeps the
// strided stage writes free of bank conflicts.
__device__ __forceinline__ int pad16(int idx) { return idx + (idx >> 4); }

// Shared-memory view of one transform / one column: element idx lives at
// base[pad16(idx) * stride].  stride = 1 for contiguous transforms, C for a
// tile of C interleaved columns (column c at base = tile + c).
template <typename V> struct SmemView {
  V *base;
  int stride;
  __device__ __forceinline__ V ld(int idx) const { return base[pad16(idx) * stride]; }
  __device__ __forceinline__ void st(int idx, V v) const { base[pad16(idx) * stride] = v; }
};

// Shared-memory view of one of 8 interleaved fp32 columns (or 4 fp64): each
// position is a 64-byte row of the C columns, so a warp touches 4 positions
// and two of them share each 128-byte row of banks.  Positions whose index
// differs by an even number land in the same half of that row (the radix-2
// stage's writes at 2i + v hit one half four times), so the position is
// stored at idx ^ ((idx >> 1) & 1): the half is then the parity of bits 0
// and 1, which splits every stage pattern of these transforms (four
// consecutive positions; 2i + v for four consecutive i; pairs 32 apart)
// two and two.  No padding: L slots per column.
template <typename V> struct SwzView {
  V *base;
  int stride;
  __device__ __forceinline__ static int swz(int idx) { return idx ^ ((idx >> 1) & 1); }
  __device__ __forceinline__ V ld(int idx) const { return base[swz(idx) * stride]; }
  __device__ __forceinline__ void st(int idx, V v) const { base[swz(idx) * stride] = v; }
};

// One radix-R Stockham stage on the registers of thread t.  x[w] holds
// element t + w*TP of the stage input.  Butterfly s (< E/R) is
// i = t + s*TP; its inputs are x[s + u*(E/R)] and its outputs go back to the
// same registers.  m = 2^LOGM is the previous block length (twiddle
// W_{R m}^{(i mod m) u} on input u).
// With a twiddle table (tw != nullptr, this stage's part of it) the
// twiddles are read from it instead of computed.
template <int R, int E, int TP, int LOGM, int DIR, bool TABLE, typename V>
__device__ __forceinline__ void stage_compute(V *x, int t, const V *tw) {
  constexpr int S = E / R;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    V y[R];
#pragma unroll
    for (int u = 0; u < R; ++u) y[u] = x[s + u * S];
    if constexpr (LOGM > 0) {
      using T = decltype(V::x);
      constexpr int M = 1 << LOGM;
      const int i = t + s * TP;
      const int p = i & (M - 1);
      if constexpr (TABLE) {
#pragma unroll
        for (int u = 1; u < R; ++u) y[u] = c_mul(y[u], tw[u * M + p]);
      } else {
        V w = twiddle<DIR>((long long)p, LOGM + ilog2(R), T());
        V pw[R];
        powers<R>(w, pw);
#pragma unroll
        for (int u = 1; u < R; ++u) y[u] = c_mul(y[u], pw[u]);
      }
    }
    dft_reg<R, DIR>(y);
#pragma unroll
    for (int v = 0; v < R; ++v) x[s + v * S] = y[v];
  }
}

// Write the outputs of stage (R, m) to shared memory at their Stockham
// positions q*R*m + p + v*m (i = q*m + p).
template <int R, int E, int TP, int LOGM, typename V, class View>
__device__ __forceinline__ void stage_store(const V *x, int t, const View &sm) {
  constexpr int S = E / R;
  constexpr int M = 1 << LOGM;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int i = t + s * TP;
    const int q = i >> LOGM, p = i & (M - 1);
    const int base = q * R * M + p;
#pragma unroll
    for (int v = 0; v < R; ++v) sm.st(base + v * M, x[s + v * S]);
  }
}

// Barriers between the stages: the whole block (default), or a named
// barrier of the `count` threads that share one transform (bar.sync id,
// count), so that several independent transforms in a block do not wait
// for one another.
struct BlockSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
struct GroupSync {
  int id;     // 1 .. 15 (0 is the block-wide barrier)
  int count;  // threads of the group, a multiple of 32
  __device__ __forceinline__ void operator()() const {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
  }
};

template <int LOGL, int K, int DIR, bool TABLE, bool SYNC_FIRST, typename V, class View,
          class Sync = BlockSync>
__device__ __forceinline__ void run_stages(V *x, int t, const View &sm, const V *tw,
                                           Sync sync = Sync()) {
  using P = StagePlan<LOGL>;
  if constexpr (K < P::NS) {
    constexpr int R = P::radix(K);
    constexpr int LOGM = P::log_m(K);
    if constexpr (K > 0) {
#pragma unroll
      for (int w = 0; w < P::E; ++w) x[w] = sm.ld(t + w * P::TP);
    }
    stage_compute<R, P::E, P::TP, LOGM, DIR, TABLE>(x, t, TABLE ? tw + P::tw_offset(K) : tw);
    if constexpr (K + 1 < P::NS) {
      // Everyone has read the previous stage's data (for the first stage:
      // whatever the caller last read from this shared memory).
      if constexpr (K > 0 || SYNC_FIRST) sync();
      stage_store<R, P::E, P::TP, LOGM>(x, t, sm);
      sync();  // this stage's data is complete
    }
    run_stages<LOGL, K + 1, DIR, TABLE, SYNC_FIRST>(x, t, sm, tw, sync);
  }
}

// The whole on-chip transform of length 2^LOGL.  On entry x[w] is element
// t + w*TP of the input (natural order); on exit x[w] is element t + w*TP of
// its DFT (natural order).  Every thread of the block must call this the
// same number of times (it contains __syncthreads when L > 16).  With
// TABLE, the stage twiddles come from `tw` (filled by fill_twiddle_table).
// SYNC_FIRST = false drops the barrier before the first stage's shared-memory
// writes: for callers that have not read `sm` since their last barrier (a
// transform loaded from global memory, or from `sm` before a barrier).
template <int LOGL, int DIR, bool TABLE = false, bool SYNC_FIRST = true, typename V,
          class View = SmemView<V>, class Sync = BlockSync>
__device__ __forceinline__ void fft_on_chip(V *x, int t, const View &sm, const V *tw = nullptr,
                                            Sync sync = Sync()) {
  run_stages<LOGL, 0, DIR, TABLE, SYNC_FIRST>(x, t, sm, tw, sync);
}

// Fills the stage-twiddle table of an on-chip transform of length 2^LOGL
// (StagePlan::TW_ELEMS entries), each entry from one accurate evaluation.
// Threads tid = 0 .. nthreads-1 of the block share the work; the caller
// synchronises before use.
template <int LOGL, int DIR, typename V>
__device__ __forceinline__ void fill_twiddle_table(V *tw, int tid, int nthreads) {
  using P = StagePlan<LOGL>;
  using T = decltype(V::x);
  for (int k = 1; k < P::NS; ++k) {
    const int R = P::radix(k), lm = P::log_m(k), M = 1 << lm;
    V *dst = tw + P::tw_offset(k);
    for (int e = tid; e < R * M; e += nthreads) {
      const int u = e >> lm, p = e & (M - 1);
      dst[e] = twiddle<DIR>((long long)p * u, lm + ilog2(R), T());
    }
  }
}

// x[w] *= a * s^w for w < E (the inter-pass twiddle of one thread's
// elements): the factors a s^w are built as a, a s, a s^2, a s^3 and then
// stepped by s^4, at most five products deep.
template <int E, typename V> __device__ __forceinline__ void apply_geometric(V *x, V a, V s) {
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
        x[4 * blk + j] = c_mul(x[4 * blk + j], q[j]);
        if (blk + 1 < E / 4) q[j] = c_mul(q[j], s4);
      }
    }
  } else {
    V pw[E];
    powers<E>(s, pw);
#pragma unroll
    for (int w = 0; w < E; ++w) x[w] = c_mul(x[w], c_mul(a, pw[w]));
  }
}

}  // namespace fftgb
