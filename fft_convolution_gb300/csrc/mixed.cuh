// mixed.cuh -- on-chip mixed-radix transforms for lengths
// N = 2^a 3^b 5^c 7^d 11^e 13^f.
//
// "FFT on GPU" (section Algorithm per signal Length) names the mixed-radix
// FFT for lengths such as 12 = 3 * 4 beside the power-of-two one.  The
// Stockham stage of "Stockham FFT Butterfly Algorithm in Parallel GLSL"
// (section Stockham) holds for any radix R once the block length m is the
// product of the radices before it:
//   out[q R m + p + v m] = sum_{u<R} W_R^{u v} (W_{R m}^{p u} in[i + u N/R]),
//   i = q m + p,  p < m,  q < N/(R m),
// natural order in and out.  A block holds F whole transforms in shared
// memory (two buffers, one barrier per stage; the first stage reads global
// memory, the last one writes it); every stage is a loop of its 256 threads
// over the F * N/R butterflies, each loading its R inputs,
// applying the stage twiddles (read from a per-plan table of the forward
// roots, conjugated for the inverse), running the radix-R DFT in registers
// and storing the R outputs.  Radices 2, 4, 8, 16 use the power-of-two
// register DFTs; 6, 10, 12, 14, 15 and 20 the prime-factor split into two
// coprime factors (dft_pfa); 3, 5, 7, 11 and 13 pair x_u with x_{R-u}:
//   X_v = x_0 + sum_{u<=(R-1)/2} [(x_u + x_{R-u}) cos(2 pi uv/R)
//                                 + DIR i (x_u - x_{R-u}) sin(2 pi uv/R)],
// and X_{R-v} the same with the sine term negated.
#pragma once

#include "fft_device.cuh"
#include "internal.h"

namespace fftgb {
namespace {

constexpr int kMixedThreads = 256;

// cos(2 pi k / R), sin(2 pi k / R) for R = 3, 5, 7, 11, 13, 1 <= k <= (R-1)/2
// (36 significant digits, rounded to the element type at compile time).
__host__ __device__ constexpr double odd_cos(int R, int k) {
  switch (R * 16 + k) {
    case 3 * 16 + 1: return -0.5;
    case 5 * 16 + 1: return 0.309016994374947424102293417182819059;
    case 5 * 16 + 2: return -0.809016994374947424102293417182819059;
    case 7 * 16 + 1: return 0.623489801858733530525004884004239811;
    case 7 * 16 + 2: return -0.222520933956314404288902564496794759;
    case 7 * 16 + 3: return -0.900968867902419126236102319507445051;
    case 11 * 16 + 1: return 0.841253532831181168861811648919367718;
    case 11 * 16 + 2: return 0.415415013001886425529274149229623204;
    case 11 * 16 + 3: return -0.142314838273285140443792668616369669;
    case 11 * 16 + 4: return -0.654860733945285064056925072466293553;
    case 11 * 16 + 5: return -0.959492973614497389890368057066327699;
    case 13 * 16 + 1: return 0.885456025653209895900375522015098879;
    case 13 * 16 + 2: return 0.568064746731155802511807559127516624;
    case 13 * 16 + 3: return 0.120536680255323053349067687452543582;
    case 13 * 16 + 4: return -0.354604887042535625969637892600018474;
    case 13 * 16 + 5: return -0.748510748171101098634630599701351384;
    case 13 * 16 + 6: return -0.970941817426052027156982276293789227;
    default: return 0.0;
  }
}
__host__ __device__ constexpr double odd_sin(int R, int k) {
  switch (R * 16 + k) {
    case 3 * 16 + 1: return 0.866025403784438646763723170752936183;
    case 5 * 16 + 1: return 0.951056516295153572116439333379382143;
    case 5 * 16 + 2: return 0.587785252292473129168705954639072769;
    case 7 * 16 + 1: return 0.781831482468029808708444526674057750;
    case 7 * 16 + 2: return 0.974927912181823607018131682993931217;
    case 7 * 16 + 3: return 0.433883739117558120475768332848358755;
    case 11 * 16 + 1: return 0.540640817455597582107635954318691695;
    case 11 * 16 + 2: return 0.909631995354518371411715383079028460;
    case 11 * 16 + 3: return 0.989821441880932732376092037776718787;
    case 11 * 16 + 4: return 0.755749574354258283774035843972344420;
    case 11 * 16 + 5: return 0.281732556841429697711417915346616899;
    case 13 * 16 + 1: return 0.464723172043768545656015335133104778;
    case 13 * 16 + 2: return 0.822983865893656394579617423439381991;
    case 13 * 16 + 3: return 0.992708874098053992800751649492520179;
    case 13 * 16 + 4: return 0.935016242685414823439784599837830729;
    case 13 * 16 + 5: return 0.663122658240795202376785492666766280;
    case 13 * 16 + 6: return 0.239315664287557767148753726260211895;
    default: return 0.0;
  }
}

// In-register DFT of odd prime length R (3, 5, 7, 11, 13), natural order.
template <int R, int DIR, typename V> __device__ __forceinline__ void dft_odd(V *x) {
  using T = decltype(V::x);
  constexpr int H = (R - 1) / 2;
  V s[H], d[H];
  V x0 = x[0];
  V sum = x[0];
#pragma unroll
  for (int u = 1; u <= H; ++u) {
    s[u - 1] = c_add(x[u], x[R - u]);
    d[u - 1] = c_sub(x[u], x[R - u]);
    sum = c_add(sum, s[u - 1]);
  }
  x[0] = sum;
#pragma unroll
  for (int v = 1; v <= H; ++v) {
    V a = x0, b = make_c<V>((T)0, (T)0);
#pragma unroll
    for (int u = 1; u <= H; ++u) {
      const int k = (u * v) % R;  // constant once the loops are unrolled
      const int kk = k <= H ? k : R - k;
      const T c = (T)odd_cos(R, kk);
      const T sn = (T)(k <= H ? odd_sin(R, kk) : -odd_sin(R, kk));
      a.x += s[u - 1].x * c;
      a.y += s[u - 1].y * c;
      b.x += d[u - 1].x * sn;
      b.y += d[u - 1].y * sn;
    }
    // DIR i b
    const V ib = DIR < 0 ? make_c<V>(b.y, -b.x) : make_c<V>(-b.y, b.x);
    x[v] = c_add(a, ib);
    x[R - v] = c_sub(a, ib);
  }
}

// (a^-1 mod m) for coprime a, m (compile time).
__host__ __device__ constexpr int inv_mod(int a, int m) {
  for (int x = 1; x < m; ++x)
    if ((a * x) % m == 1) return x;
  return 1;
}

template <int R, int DIR, typename V> __device__ __forceinline__ void dft_any(V *x);

// In-register DFT of length R = R1 * R2, R1 and R2 coprime, by the
// prime-factor (Good-Thomas) mapping: with input index
// u = (R2 n1 + R1 n2) mod R and output index v = (e1 k1 + e2 k2) mod R,
// e1 = R2 (R2^-1 mod R1), e2 = R1 (R1^-1 mod R2), the exponent is
//   u v = R2 e1 n1 k1 + R1 e2 n2 k2 (mod R),
// and W_R^{R2 e1 n1 k1} = W_{R1}^{n1 k1}, W_R^{R1 e2 n2 k2} = W_{R2}^{n2 k2},
// so X_v = sum_{n2} W_{R2}^{n2 k2} sum_{n1} W_{R1}^{n1 k1} x_u: R2 DFTs of
// length R1, then R1 of length R2, with no twiddle between them; the index
// maps are register renaming only (15 = 3 * 5: u = (5 n1 + 3 n2) mod 15,
// v = (10 k1 + 6 k2) mod 15).
template <int R1, int R2, int DIR, typename V> __device__ __forceinline__ void dft_pfa(V *x) {
  constexpr int R = R1 * R2;
  constexpr int E1 = R2 * inv_mod(R2 % R1, R1);
  constexpr int E2 = R1 * inv_mod(R1 % R2, R2);
  V a[R2][R1];
#pragma unroll
  for (int n2 = 0; n2 < R2; ++n2)
#pragma unroll
    for (int n1 = 0; n1 < R1; ++n1) a[n2][n1] = x[(R2 * n1 + R1 * n2) % R];
#pragma unroll
  for (int n2 = 0; n2 < R2; ++n2) dft_any<R1, DIR>(a[n2]);
  V b[R1][R2];
#pragma unroll
  for (int k1 = 0; k1 < R1; ++k1)
#pragma unroll
    for (int n2 = 0; n2 < R2; ++n2) b[k1][n2] = a[n2][k1];
#pragma unroll
  for (int k1 = 0; k1 < R1; ++k1) dft_any<R2, DIR>(b[k1]);
#pragma unroll
  for (int k1 = 0; k1 < R1; ++k1)
#pragma unroll
    for (int k2 = 0; k2 < R2; ++k2) x[(E1 * k1 + E2 * k2) % R] = b[k1][k2];
}

// The stage radices: powers of two up to 16 (dft_reg), odd primes up to
// 13 (dft_odd) and the coprime products 6, 10, 12, 14, 15, 20 (dft_pfa).
template <int R, int DIR, typename V> __device__ __forceinline__ void dft_any(V *x) {
  if constexpr (R == 3 || R == 5 || R == 7 || R == 11 || R == 13) dft_odd<R, DIR>(x);
  else if constexpr (R == 6) dft_pfa<2, 3, DIR>(x);
  else if constexpr (R == 10) dft_pfa<2, 5, DIR>(x);
  else if constexpr (R == 12) dft_pfa<4, 3, DIR>(x);
  else if constexpr (R == 14) dft_pfa<2, 7, DIR>(x);
  else if constexpr (R == 15) dft_pfa<3, 5, DIR>(x);
  else if constexpr (R == 20) dft_pfa<4, 5, DIR>(x);
  else dft_reg<R, DIR>(x);
}

// floor(x / d) from the host-computed magic of d (exact while x * d < 2^32;
// x < F N / 2 and d <= N keep every use far below that).
__device__ __forceinline__ int div_magic(int x, int d, unsigned magic) {
  return d == 1 ? x : (int)__umulhi((unsigned)x, magic);
}

// One stage of radix R over the F transforms of a block: src and dst hold
// F transforms of N values each (stride N).  tw: this stage's table,
// W_{Rm}^{p u} (forward) at (u - 1) m + p.  The last stage writes the
// block's valid rows (`rows` of them) straight to global memory with the
// scale; the others go from one shared buffer to the other.
template <int R, int DIR, bool LAST, typename V>
__device__ __forceinline__ void mixed_stage(const V *src, V *dst, const MixedStages &ms, int k,
                                            const V *tw, int rows, decltype(V::x) scale) {
  using T = decltype(V::x);
  const int N = ms.N, m = ms.m[k];
  const int nb = N / R;
  const int total = ms.F * nb;
  const bool qfast = !LAST && ((ms.qorder >> k) & 1u);
  for (int b = threadIdx.x; b < total; b += kMixedThreads) {
    const int f = div_magic(b, nb, ms.nb_magic[k]), j = b - f * nb;
    int q, p;
    if (qfast) {  // j = p * nq + q: a warp's stores at the odd stride R m
      p = div_magic(j, ms.nq[k], ms.q_magic[k]);
      q = j - p * ms.nq[k];
    } else {      // j = q * m + p: runs of m consecutive stores
      q = div_magic(j, m, ms.m_magic[k]);
      p = j - q * m;
    }
    const int i = q * m + p;
    const V *s = src + f * N;
    V y[R];
#pragma unroll
    for (int u = 0; u < R; ++u) y[u] = s[i + u * nb];
    if (m > 1) {
#pragma unroll
      for (int u = 1; u < R; ++u) {
        const V w = __ldg(tw + (u - 1) * m + p);
        y[u] = DIR < 0 ? c_mul(y[u], w) : make_c<V>(y[u].x * w.x + y[u].y * w.y,
                                                      y[u].y * w.x - y[u].x * w.y);
      }
    }
    dft_any<R, DIR>(y);
    V *d = dst + f * N + q * R * m + p;
    if (LAST) {
      if (f < rows) {
#pragma unroll
        for (int v = 0; v < R; ++v) d[v * m] = c_scale(y[v], scale);
      }
    } else {
#pragma unroll
      for (int v = 0; v < R; ++v) d[v * m] = y[v];
    }
  }
}

template <int DIR, bool LAST, typename V>
__device__ __forceinline__ void mixed_stage_any(const V *src, V *dst, const MixedStages &ms,
                                                int k, const V *tw, int rows,
                                                decltype(V::x) scale) {
  const V *t = tw + ms.tw_off[k];
  switch (ms.radix[k]) {
    case 2: mixed_stage<2, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 3: mixed_stage<3, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 4: mixed_stage<4, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 5: mixed_stage<5, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 7: mixed_stage<7, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 11: mixed_stage<11, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 13: mixed_stage<13, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 8: mixed_stage<8, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 6: mixed_stage<6, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 10: mixed_stage<10, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 12: mixed_stage<12, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 14: mixed_stage<14, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 15: mixed_stage<15, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    case 20: mixed_stage<20, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
    default: mixed_stage<16, DIR, LAST>(src, dst, ms, k, t, rows, scale); break;
  }
}

// The first stage (m = 1, no twiddles) read straight from global memory:
// butterfly i of row f takes g[f*N + i + u*nb] (consecutive threads read
// consecutive elements) and writes dst[f*N + i*R + v].  Each thread first
// loads G butterflies (G*R <= 16 fp32 / 8 fp64 values in flight), then
// computes and stores them.  Rows at or beyond `rows` read as zeros.
template <int R, int DIR, typename V>
__device__ __forceinline__ void mixed_first_stage(const V *g, V *dst, const MixedStages &ms,
                                                  int rows) {
  using T = decltype(V::x);
  constexpr int MAXV = sizeof(T) == 4 ? 16 : 8;
  constexpr int G = 4 * R <= MAXV ? 4 : (2 * R <= MAXV ? 2 : 1);
  const int N = ms.N, nb = N / R;
  const int total = ms.F * nb;
  for (int b0 = threadIdx.x; b0 < total; b0 += G * kMixedThreads) {
    V y[G][R];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int b = b0 + j * kMixedThreads;
      const int f = div_magic(b, nb, ms.nb_magic[0]), i = b - f * nb;
      const bool live = b < total && f < rows;
      const V *s = g + (long long)f * N + i;
#pragma unroll
      for (int u = 0; u < R; ++u) y[j][u] = live ? s[u * nb] : make_c<V>((T)0, (T)0);
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int b = b0 + j * kMixedThreads;
      if (b < total) {
        const int f = div_magic(b, nb, ms.nb_magic[0]), i = b - f * nb;
        dft_any<R, DIR>(y[j]);
        V *d = dst + f * N + i * R;
#pragma unroll
        for (int v = 0; v < R; ++v) d[v] = y[j][v];
      }
    }
  }
}

template <int DIR, typename V>
__device__ __forceinline__ void mixed_first_stage_any(const V *g, V *dst, const MixedStages &ms,
                                                      int rows) {
  switch (ms.radix[0]) {
    case 2: mixed_first_stage<2, DIR>(g, dst, ms, rows); break;
    case 3: mixed_first_stage<3, DIR>(g, dst, ms, rows); break;
    case 4: mixed_first_stage<4, DIR>(g, dst, ms, rows); break;
    case 5: mixed_first_stage<5, DIR>(g, dst, ms, rows); break;
    case 7: mixed_first_stage<7, DIR>(g, dst, ms, rows); break;
    case 11: mixed_first_stage<11, DIR>(g, dst, ms, rows); break;
    case 13: mixed_first_stage<13, DIR>(g, dst, ms, rows); break;
    case 8: mixed_first_stage<8, DIR>(g, dst, ms, rows); break;
    case 6: mixed_first_stage<6, DIR>(g, dst, ms, rows); break;
    case 10: mixed_first_stage<10, DIR>(g, dst, ms, rows); break;
    case 12: mixed_first_stage<12, DIR>(g, dst, ms, rows); break;
    case 14: mixed_first_stage<14, DIR>(g, dst, ms, rows); break;
    case 15: mixed_first_stage<15, DIR>(g, dst, ms, rows); break;
    case 20: mixed_first_stage<20, DIR>(g, dst, ms, rows); break;
    default: mixed_first_stage<16, DIR>(g, dst, ms, rows); break;
  }
}

template <typename T, int DIR>
__global__ void __launch_bounds__(kMixedThreads, sizeof(T) == 4 ? 4 : 2)
    mixed_rows_kernel(const vec2_t<T> *in, vec2_t<T> *out, long long batch, MixedStages ms,
                      const vec2_t<T> *__restrict__ tw, T scale) {
  using V = vec2_t<T>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V *cur = reinterpret_cast<V *>(smem_raw);
  V *nxt = cur + ms.F * ms.N;
  const long long row0 = (long long)blockIdx.x * ms.F;
  const long long left = batch - row0;
  const int rows = left < ms.F ? (int)left : ms.F;
  // The first stage straight from global memory into shared memory, the
  // middle stages between the two shared buffers (one barrier each: a
  // stage's output is complete and its input buffer free for the next
  // output), the last stage to global memory.  (Persistent blocks
  // prefetching the next rows into a third buffer measured slower: one
  // block fewer per SM.)
  // Programmatic dependent launch, as the row kernel: wait for the
  // previous kernel before the first stage reads global memory; the next
  // kernel may be scheduled once this block has its data on chip.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  mixed_first_stage_any<DIR>(in + row0 * ms.N, cur, ms, rows);
  asm volatile("griddepcontrol.launch_dependents;");
  __syncthreads();
  const int S = ms.nstages;  // >= 2 for every planned length (N > 64, R <= 16)
  for (int k = 1; k < S - 1; ++k) {
    mixed_stage_any<DIR, false>(cur, nxt, ms, k, tw, rows, (T)1);
    __syncthreads();
    V *tmp = cur;
    cur = nxt;
    nxt = tmp;
  }
  mixed_stage_any<DIR, true>(cur, out + row0 * ms.N, ms, S - 1, tw, rows, scale);
}

template <typename T>
cudaError_t mixed_exec_t(const void *in, void *out, long long batch, const MixedStages &ms,
                         const void *tw, int dir, cudaStream_t st) {
  using V = vec2_t<T>;
  const size_t smem = 2 * (size_t)ms.F * ms.N * sizeof(V);
  auto kern = dir < 0 ? mixed_rows_kernel<T, -1> : mixed_rows_kernel<T, 1>;
  if (smem > 48 * 1024) {
    // The largest size any plan needs, once per device and direction.
    static DeviceOnce attr_set[2];
    const size_t max_smem = 2 * (size_t)(sizeof(T) == 4 ? kMixedMaxF32 : kMixedMaxF64) * sizeof(V);
    const cudaError_t e = smem_limit_once((const void *)kern, max_smem, attr_set[dir < 0 ? 0 : 1]);
    if (e != cudaSuccess) return e;
  }
  const long long grid = (batch + ms.F - 1) / ms.F;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const T scale = dir < 0 ? (T)1 : (T)(1.0 / ms.N);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kMixedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const V *>(in), static_cast<V *>(out), batch,
                            ms, static_cast<const V *>(tw), scale);
}

}  // namespace
}  // namespace fftgb
