// fft_pass.cuh -- one HBM pass of a multi-pass transform, and the column
// pass of the 2D transform.
//
// A transform of N = 2^log_n points that does not fit on chip is split into
// passes N = L_0 L_1 ... ; pass k is one radix-L_k Stockham stage (the stage
// of "Stockham FFT Butterfly Algorithm in Parallel GLSL", items 2-3, with
// radix L_k instead of 2 -- see fft_device.cuh) whose L_k-point butterflies
// are themselves whole on-chip transforms.  With previous block length m:
//   butterfly i = q*m + p reads      in[i + u*N/L],            u < L
//   multiplies input u by           W_{L m}^{p u}               (m > 1)
//   and writes                       out[q*L*m + p + v*m],     v < L.
// The first pass (m = 1) writes out[i*L + v]: a tile's results form one
// contiguous block, which is staged through shared memory so that the HBM
// writes stay coalesced.  The last pass (L*m = N) reads and writes the same
// positions, so it may run in place.
//
// The 2D column pass is the same kernel with N = H*W, L = H, m = W and no
// twiddle: it transforms every column of an H x W image in place.
//
// One block takes a tile of C consecutive butterflies (columns) i, so every
// HBM access moves C contiguous complex values (C * 8 or C * 16 bytes, 64 KB
// tiles: C = 16 fp32 columns for L = 512).  Within the tile column c lives in
// shared memory at pad16(idx) * C + c: the C lanes that share a row touch C
// consecutive slots, free of bank conflicts.
#pragma once

#include "fft_device.cuh"
#include "internal.h"

namespace fftgb {
// Kernels and their launchers have internal linkage: every translation unit
// that instantiates one owns its own copy, so no kernel is registered twice.
namespace {

template <typename T, int LOGL> struct PassConfig {
  using P = StagePlan<LOGL>;
  static constexpr long long TILE_BYTES_TARGET = 65536;
  static constexpr long long C_RAW =
      TILE_BYTES_TARGET / ((long long)P::L * (long long)sizeof(vec2_t<T>));
  static constexpr int C = C_RAW < 1 ? 1 : (C_RAW > 64 ? 64 : (int)C_RAW);
  static constexpr int THREADS = C * P::TP;
  // Ask for registers that let 1024 threads (two 512-thread tiles) share an
  // SM in fp32, so one tile's loads overlap another's compute and stores;
  // 512 threads in fp64 (128 registers: the 16 values a thread holds take
  // 32 registers each way, and fewer registers spill them).
  static constexpr int RESIDENT = sizeof(T) == 8 ? 512 : 1024;
  static constexpr int MIN_BLOCKS = THREADS >= RESIDENT ? 1 : RESIDENT / THREADS;
  static constexpr int ROW_ELEMS =
      P::SMEM_ELEMS > P::L + 1 ? P::SMEM_ELEMS : P::L + 1;  // exchange or transpose
  static constexpr int EXCHANGE_ELEMS = C * ROW_ELEMS;
  // Exchange space, then the stage-twiddle table shared by the tile's
  // columns -- unless the two together would not fit shared memory (fp64,
  // L = 2^13): then the stage twiddles are computed.
  static constexpr bool TABLE =
      ((size_t)EXCHANGE_ELEMS + P::TW_ELEMS) * sizeof(vec2_t<T>) <= 200 * 1024;
  static constexpr size_t SMEM =
      ((size_t)EXCHANGE_ELEMS + (TABLE ? P::TW_ELEMS : 0)) * sizeof(vec2_t<T>);
};

// Plain complex load / store (element `pos` of transform `b`).
template <typename V> struct LoadComplex {
  const V *p;
  long long bstride;
  __device__ __forceinline__ V operator()(long long b, long long pos) const {
    return p[b * bstride + pos];
  }
};
template <typename V> struct StoreComplex {
  V *p;
  long long bstride;
  __device__ __forceinline__ void operator()(long long b, long long pos, V v) const {
    p[b * bstride + pos] = v;
  }
};

// Optional two-level table of the inter-pass twiddles W_{L m}^e for this
// pass's direction: W^e = hi[e >> lo_bits] * lo[e & (2^lo_bits - 1)].
// Used where sincospi is expensive (fp64); lo == nullptr computes them.
// The tables are built for W_{2^log_size}; a pass with L m < 2^log_size
// scales its exponent up.
template <typename V> struct TwiddleTables {
  const V *lo;
  const V *hi;
  int lo_bits;
  int log_size;
};

struct PassGeom {
  int log_n;
  int log_m;
  int twiddle;
  long long grid_per_batch;  // tiles per transform (a power of two)
  long long total;           // grid_per_batch * batch: the tiles of the launch
  int log_gpb;               // log2(grid_per_batch)
};

// Persistent: each block fills the stage-twiddle table once, then walks
// the launch's tiles blockIdx.x, blockIdx.x + gridDim.x, ...
template <typename T, int LOGL, int DIR, class Load, class Store>
__global__ void __launch_bounds__(PassConfig<T, LOGL>::THREADS, PassConfig<T, LOGL>::MIN_BLOCKS)
    fft_pass_kernel(Load load, Store store, PassGeom g, TwiddleTables<vec2_t<T>> tt) {
  using V = vec2_t<T>;
  using P = StagePlan<LOGL>;
  using Cfg = PassConfig<T, LOGL>;
  constexpr int C = Cfg::C;
  constexpr int L = P::L;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V *smem = reinterpret_cast<V *>(smem_raw);
  V *twt = smem + Cfg::EXCHANGE_ELEMS;

  const int c = threadIdx.x % C;   // column within the tile
  const int t = threadIdx.x / C;   // thread within the column
  const long long cols = 1LL << (g.log_n - LOGL);  // N / L butterflies
  if constexpr (Cfg::TABLE) fill_twiddle_table<LOGL, DIR>(twt, threadIdx.x, Cfg::THREADS);
  __syncthreads();

  for (long long blk = blockIdx.x; blk < g.total; blk += gridDim.x) {
    const long long tile = blk & (g.grid_per_batch - 1);
    const long long b = blk >> g.log_gpb;
    const long long i = tile * C + c;
    const bool active = i < cols;

    V x[P::E];
    if (active) {
#pragma unroll
      for (int w = 0; w < P::E; ++w) x[w] = load(b, i + (long long)(t + w * P::TP) * cols);
      if (g.twiddle && g.log_m > 0) {
        // W_{L m}^{p u} for u = t + w*TP.
        const long long p = i & ((1LL << g.log_m) - 1);
        const int log_lm = g.log_m + LOGL;
        if (tt.lo) {
          const long long emask = (1LL << log_lm) - 1, lmask = (1LL << tt.lo_bits) - 1;
          const int up = tt.log_size - log_lm;
#pragma unroll
          for (int w = 0; w < P::E; ++w) {
            const long long e = ((p * (t + w * P::TP)) & emask) << up;
            x[w] = c_mul(x[w], c_mul(tt.hi[e >> tt.lo_bits], tt.lo[e & lmask]));
          }
        } else {
          // W^{p t} * (W^{p TP})^w.
          apply_geometric<P::E>(x, twiddle<DIR>(p * t, log_lm, T()),
                                twiddle<DIR>(p * P::TP, log_lm, T()));
        }
      }
    } else {
#pragma unroll
      for (int w = 0; w < P::E; ++w) x[w] = make_c<V>((T)0, (T)0);
    }

    const SmemView<V> sm{smem + c, C};
    // The previous tile's shared-memory reads ended before the barrier at the
    // end of the loop: the first stage needs no barrier of its own.
    fft_on_chip<LOGL, DIR, Cfg::TABLE, false>(x, t, sm, Cfg::TABLE ? twt : nullptr);

    if constexpr (DIR > 0) {
#pragma unroll
      for (int w = 0; w < P::E; ++w) x[w] = c_scale(x[w], (T)(1.0 / L));  // 1/L per pass
    }

    if (g.log_m == 0) {
      // First pass: butterfly i's outputs go to i*L + v, so the tile's outputs
      // are the contiguous block [tile*C*L, (tile+1)*C*L).  Stage them in
      // shared memory (row c padded to L+1 slots) and write linearly.
      constexpr int RS = L + 1;
      __syncthreads();
#pragma unroll
      for (int w = 0; w < P::E; ++w) smem[c * RS + t + w * P::TP] = x[w];
      __syncthreads();
      const long long base = tile * C * L;
#pragma unroll
      for (int w = 0; w < P::E; ++w) {
        const int o = threadIdx.x + w * Cfg::THREADS;
        const int cc = o / L, v = o % L;
        if (tile * C + cc < cols) store(b, base + o, smem[cc * RS + v]);
      }
    } else if (active) {
      const long long m = 1LL << g.log_m;
      const long long q = i >> g.log_m, p = i & (m - 1);
      const long long base = q * L * m + p;
#pragma unroll
      for (int w = 0; w < P::E; ++w) store(b, base + (long long)(t + w * P::TP) * m, x[w]);
    }
    __syncthreads();  // shared memory is free for the next tile
  }
}

// Tiles (of C consecutive butterflies) a pass with on-chip length 2^log_l
// has per transform.
template <typename T, int LOGL> long long pass_tiles(int log_n) {
  const long long cols = 1LL << (log_n - LOGL);
  return (cols + PassConfig<T, LOGL>::C - 1) / PassConfig<T, LOGL>::C;
}

template <typename T, int LOGL, int DIR, class Load, class Store>
cudaError_t launch_pass_t(Load load, Store store, int log_n, int log_m, int twiddle,
                          long long batch, cudaStream_t st,
                          TwiddleTables<vec2_t<T>> tt = {nullptr, nullptr, 0, 0}) {
  using C = PassConfig<T, LOGL>;
  auto kern = fft_pass_kernel<T, LOGL, DIR, Load, Store>;
  if (C::SMEM > 48 * 1024) {
    static DeviceOnce attr_set;
    const cudaError_t e = smem_limit_once((const void *)kern, C::SMEM, attr_set);
    if (e != cudaSuccess) return e;
  }
  const long long tiles = pass_tiles<T, LOGL>(log_n);
  int log_gpb = 0;
  while ((1LL << log_gpb) < tiles) ++log_gpb;
  PassGeom g{log_n, log_m, twiddle, tiles, tiles * batch, log_gpb};
  if (g.total <= 0) return cudaErrorInvalidConfiguration;
  // Persistent grid: as many blocks as fit on the device at once.
  static std::atomic<int> occupancy[64];
  const int per_sm = blocks_per_sm_once((const void *)kern, C::THREADS, C::SMEM, occupancy);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long grid = (long long)(per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
  if (grid > g.total) grid = g.total;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, st>>>(load, store, g, tt);
  return cudaGetLastError();
}

template <typename T, int LOGL, int DIR, bool SHFL = false>
cudaError_t launch_pass_tma_t(const void *in, void *out, int log_n, int log_m, int twiddle,
                              long long batch, cudaStream_t st, int overlap = 0);
template <typename T, int LOGL, int DIR>
cudaError_t launch_pass_cluster_t(const void *in, void *out, int log_n, int log_m, int twiddle,
                                  long long batch, cudaStream_t st, int debug_fail = 0,
                                  unsigned poll_limit = 0);

template <typename T, int DIR, int MAXLOG, int LOGL = 1>
cudaError_t dispatch_pass(const PassArgs &a, const void *in, void *out, cudaStream_t st) {
  if constexpr (LOGL > MAXLOG) {
    return cudaErrorInvalidValue;
  } else {
    if (a.log_l == LOGL) {
      using V = vec2_t<T>;
      const long long n = 1LL << a.log_n;
      cudaError_t e = launch_pass_cluster_t<T, LOGL, DIR>(in, out, a.log_n, a.log_m, a.twiddle,
                                                          a.batch, st);
      if (e != cudaErrorNotSupported) return e;
      e = launch_pass_tma_t<T, LOGL, DIR>(in, out, a.log_n, a.log_m, a.twiddle, a.batch, st,
                                          a.overlap);
      if (e != cudaErrorNotSupported) return e;
      return launch_pass_t<T, LOGL, DIR>(LoadComplex<V>{static_cast<const V *>(in), n},
                                         StoreComplex<V>{static_cast<V *>(out), n}, a.log_n,
                                         a.log_m, a.twiddle, a.batch, st);
    }
    return dispatch_pass<T, DIR, MAXLOG, LOGL + 1>(a, in, out, st);
  }
}

}  // namespace
}  // namespace fftgb
