// fft_pass_tma.cuh -- the HBM pass kernel of fft_pass.cuh with its strided
// tiles moved by the Tensor Memory Accelerator.
//
// Same computation as fft_pass_kernel (one radix-L Stockham stage over HBM
// whose L-point butterflies are on-chip transforms of C consecutive
// columns), organised for sm_103a:
//   * persistent blocks (as many as fit per SM), each walking the tiles
//     blockIdx.x, blockIdx.x + gridDim.x, ...;
//   * the input tile (L rows x C columns, rows 8*cols bytes apart) arrives
//     by cp.async.bulk.tensor into one of up to three shared-memory buffers,
//     tracked by an mbarrier, up to two tiles ahead of the one the block
//     computes -- HBM reads overlap the arithmetic inside one block and the
//     load/store units carry only the shared-memory exchanges;
//   * outputs of passes with m > 1 (rows m elements apart) leave by a TMA
//     tensor store from the same buffer; the first pass (m = 1), whose tile
//     output is one contiguous block, stages it column by column and
//     writes each column's L values with one bulk copy.
// Every mbarrier wait is bounded: a wait that runs out records
// kDeviceErrorTimeout in the device status word and the block stops
// (fft_device_status reports it).
#pragma once

#include <cuda.h>

#include <type_traits>

#include "fft_pass.cuh"
#include "fft_warp.cuh"

namespace fftgb {

constexpr int kDeviceErrorTimeout = 1;

namespace {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait: false if the phase did not complete within `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          uint32_t limit = 1u << 22) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int x, int y,
                                             int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group"
      " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// Contiguous shared -> global copy by the bulk-copy engine (both addresses
// 16-byte aligned, size a multiple of 16), tracked by the bulk group.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// SHFL: the warp-shuffle variant of the 512-point fp32 pass (one warp per
// column, fft512_warp; see the kernel).
template <typename T, int LOGL, bool SHFL = false> struct TmaConfig {
  using P = StagePlan<LOGL>;
  using V = vec2_t<T>;
  static constexpr int L = P::L;
  // Half the plain kernel's tile width, but rows of at least 32 bytes:
  // several double-buffered blocks per SM, whose barrier waits and compute
  // overlap.  Measured on GB300 (2^26 fp32, L = 512): 16 columns, one block
  // per SM 0.71 ms; 8 columns, three blocks 0.61 ms; 4 columns 0.76 ms.  At
  // L = 2048 (4 columns = 32 bytes) the width stays.
  static constexpr int C_MIN = (int)(32 / sizeof(V));
  static constexpr int C = PassConfig<T, LOGL>::C / 2 >= C_MIN
                               ? PassConfig<T, LOGL>::C / 2
                               : (PassConfig<T, LOGL>::C < C_MIN ? PassConfig<T, LOGL>::C : C_MIN);
  static constexpr int THREADS = C * P::TP;
  static constexpr int ROWS_PER_BOX = L < 256 ? L : 256;  // TMA box limit per dimension
  static constexpr int BOXES = L / ROWS_PER_BOX;
  static constexpr uint32_t TILE_BYTES = (uint32_t)(C * L * sizeof(V));
  // First-pass staging stride: column c at c * RS.  RS - L = 32 / C (the
  // rows one warp covers) spreads the writes of a warp's lanes evenly over
  // the banks; at least 2 for fp32, so every column starts 16-byte aligned.
  static constexpr int PAD = 32 / C >= 2 ? 32 / C : (sizeof(T) == 4 ? 2 : 1);
  static constexpr int RS = L + PAD;
  // Exchange layout: 64-byte rows of C columns take the swizzled view
  // (SwzView, L slots per column) when the transform starts with a radix-2
  // stage (whose writes land at 2i + v: the pattern the swizzle balances);
  // other tiles the padded one (which balances a first stage's 16i + v).
  static constexpr bool SWIZZLE = C * sizeof(V) == 64 && P::R0 == 2;
  // The shuffle variant exists for one warp of 32 lanes x 16 values per
  // column and 64-byte tile rows: fp32, L = 512, C = 8.
  static constexpr bool SHFL_OK = std::is_same<T, float>::value && LOGL == 9 && C == 8;
  static_assert(!SHFL || SHFL_OK, "warp-shuffle pass: fp32, 512 points, 8 columns");
  static constexpr int RAW_EX =
      SHFL || SWIZZLE ? L * C : PassConfig<T, LOGL>::ROW_ELEMS * C;
  static constexpr int RAW_ELEMS = RAW_EX > C * RS ? RAW_EX : C * RS;
  static constexpr int MIN_BLOCKS = THREADS >= 1024 ? 1 : (THREADS >= 512 ? 2 : (THREADS >= 256 ? 3 : 4));
  // Buffers start on 128-byte boundaries (TMA), 1024-byte ones for the
  // swizzled tiles of the shuffle variant (whose pattern follows address
  // bits 4..8 within each 512-byte span).
  static constexpr int ALIGN = SHFL ? 1024 : 128;
  static constexpr int BUF_ELEMS =
      ((RAW_ELEMS * (int)sizeof(V) + ALIGN - 1) / ALIGN) * ALIGN / (int)sizeof(V);
  // Stage-twiddle table shared by the block's columns (rounded to 128 B);
  // the shuffle variant forms its twiddles in registers.
  static constexpr int TW_ELEMS =
      SHFL ? 0 : ((P::TW_ELEMS * (int)sizeof(V) + 127) / 128) * 128 / (int)sizeof(V);
  // Barriers and twiddle table before the buffers, rounded to ALIGN.
  static constexpr int HEAD =
      ((128 + TW_ELEMS * (int)sizeof(V) + ALIGN - 1) / ALIGN) * ALIGN;
  // Buffers per block: the loads run NBUF - 1 tiles ahead of the
  // computation.  Three (two tiles in flight) when that leaves room for two
  // blocks per SM, else two when three blocks still fit, else one (the
  // overlap then comes from the other blocks on the SM).  Measured on GB300
  // (fp32, ms): 2^26 transform 0.570 with two buffers at three blocks per SM,
  // 0.542 with three at two blocks, 0.831 with four at one block; 8 x 2048^2
  // forward + inverse 0.415, 0.397, 0.487.
  static constexpr int NBUF = 3 * BUF_ELEMS * sizeof(V) <= 110 * 1024
                                  ? 3
                                  : (2 * BUF_ELEMS * sizeof(V) <= 76 * 1024 ? 2 : 1);
  static constexpr size_t SMEM = ALIGN + HEAD + NBUF * (size_t)BUF_ELEMS * sizeof(V);
};

// Byte offset within a tile of 64-byte rows as the TMA's 64-byte swizzle
// places it: the 16-byte chunk index (bits 4..5) is XORed with bits 7..8
// (the row index halved, mod 4), for a tile starting on a 512-byte boundary.
__device__ __forceinline__ int swz64(int o) { return o ^ (((o >> 7) & 3) << 4); }

struct TmaGeom {
  int log_n;
  int log_m;
  int twiddle;
  long long tiles_per_batch;
  long long total_tiles;
  // Test hook of the cluster kernel (0 in every transform): block rank
  // debug_fail - 1 arms its first tile load for 16 bytes that never come
  // (and issues no copy); its waits give up after poll_limit polls.
  int debug_fail;
  unsigned poll_limit;
  int log_tpb;  // log2(tiles_per_batch): tile counts are powers of two
};

// log2 of a power of two (host).
inline int log2_pow2(long long v) {
  int l = 0;
  while ((1LL << l) < v) ++l;
  return l;
}

// SHFL (fp32, L = 512, 8 columns; FFT_OPT_PASS_SHFL): warp w transforms
// column w of the tile by fft512_warp -- lane l holds rows l + 32 r --
// exchanging by __shfl_xor_sync instead of through shared memory.  The tile
// arrives and leaves with the TMA's 64-byte swizzle, which keeps a warp's
// accesses to one column within 4 shared-memory wavefronts (16 without it);
// each warp reads and writes only its own column's slots, so two block
// barriers per tile remain (after the loads, before the store) instead of
// six.
template <typename T, int LOGL, int DIR, bool SHFL = false>
__global__ void __launch_bounds__(TmaConfig<T, LOGL, SHFL>::THREADS,
                                  TmaConfig<T, LOGL, SHFL>::MIN_BLOCKS)
    fft_pass_tma_kernel(const __grid_constant__ CUtensorMap tin,
                        const __grid_constant__ CUtensorMap tout, vec2_t<T> *out_linear,
                        TmaGeom g, int *status) {
  using Cfg = TmaConfig<T, LOGL, SHFL>;
  using P = StagePlan<LOGL>;
  using V = vec2_t<T>;
  constexpr int C = Cfg::C;
  constexpr int L = Cfg::L;
  constexpr unsigned A = Cfg::ALIGN;
  extern __shared__ __align__(128) unsigned char smem_tma[];
  // TMA destinations must be 128-byte aligned (1024 for the swizzled
  // tiles): round the base up (the allocation carries ALIGN spare bytes).
  unsigned char *base = smem_tma + ((A - (smem_addr(smem_tma) & (A - 1))) & (A - 1));
  uint64_t *bar = reinterpret_cast<uint64_t *>(base);
  V *const twt = reinterpret_cast<V *>(base + 128);
  V *const buf0 = reinterpret_cast<V *>(base + Cfg::HEAD);

  const int tid = threadIdx.x;
  const int c = tid % C;
  const int t = tid / C;

  auto issue_load = [&](long long tile, int s) {
    const long long b = tile >> g.log_tpb;
    const long long i0 = (tile & (g.tiles_per_batch - 1)) * C;
    V *dst = buf0 + s * Cfg::BUF_ELEMS;
    mbar_expect_tx(&bar[s], Cfg::TILE_BYTES);
#pragma unroll
    for (int k = 0; k < Cfg::BOXES; ++k)
      tma_load_3d(dst + k * Cfg::ROWS_PER_BOX * C, &tin, &bar[s], (int)(2 * i0),
                  k * Cfg::ROWS_PER_BOX, (int)b);
  };

  constexpr int NB = Cfg::NBUF;
  static_assert(NB >= 1 && NB <= 15, "one mbarrier per buffer in the first 128 bytes");
  if (tid == 0) {
#pragma unroll
    for (int j = 0; j < NB; ++j) mbar_init(&bar[j], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if constexpr (!SHFL) fill_twiddle_table<LOGL, DIR>(twt, tid, Cfg::THREADS);
  __syncthreads();
  // When launched with programmatic dependent launch (after another pass)
  // the set-up above overlaps the previous kernel's tail; every global
  // access (the TMA loads and the stores, all issued below) waits for that
  // kernel's completion here (without it the wait returns at once).  No
  // early trigger for the next kernel: a following 2D row kernel, scheduled
  // early, slowed the 8 x 2048^2 step from 0.379 to 0.424 ms; the trigger
  // at exit keeps the pass-to-pass gain (2^26: 0.535 -> 0.529 ms).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // With NB buffers the loads run NB - 1 tiles ahead of the computation:
  // tile k of this block lives in buffer k mod NB.
  if (NB > 1 && tid == 0) {
#pragma unroll
    for (int j = 0; j + 1 < NB; ++j) {
      const long long tj = blockIdx.x + (long long)j * gridDim.x;
      if (tj < g.total_tiles) issue_load(tj, j);
    }
  }

  static_assert(C <= 32, "the threads that issue bulk stores are in warp 0");
  int k = 0;
  for (long long tile = blockIdx.x; tile < g.total_tiles; tile += gridDim.x, ++k) {
    const int s = k % NB;
    V *const cur = buf0 + s * Cfg::BUF_ELEMS;
    const long long ahead = tile + (long long)(NB - 1) * gridDim.x;
    // The buffer the next load lands in, (k - 1) mod NB, last held the
    // previous tile's output: every thread finished staging it before the
    // previous iteration's last barrier, and only its bulk stores (issued by
    // threads < C, all in warp 0) may still be reading it.  So warp 0 alone
    // waits for them before thread 0 issues the load.
    if (tid < 32) {
      if (tid < C) bulk_wait_read_all();
      __syncwarp();
      if (tid == 0) {
        if (NB > 1) {
          if (ahead < g.total_tiles) issue_load(ahead, (k + NB - 1) % NB);
        } else {
          issue_load(tile, 0);
        }
      }
    }
    const bool ok = mbar_wait(&bar[s], (uint32_t)(k / NB) & 1u);

    if constexpr (SHFL) {
      const int lane = tid & 31, col = tid >> 5;
      unsigned char *const cb = reinterpret_cast<unsigned char *>(cur);
      V x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r)
        x[r] = *reinterpret_cast<const V *>(cb + swz64(((lane + 32 * r) << 6) + (col << 3)));
      if (__syncthreads_or(!ok)) {
        if (tid == 0) {
          atomicExch(status, kDeviceErrorTimeout);
#pragma unroll
          for (int j = 1; j < NB; ++j)
            if (tile + (long long)j * gridDim.x < g.total_tiles)
              mbar_wait(&bar[(k + j) % NB], (uint32_t)((k + j) / NB) & 1u);
        }
        break;
      }
      const long long b = tile >> g.log_tpb;
      const long long i0 = (tile & (g.tiles_per_batch - 1)) * C;  // the tile's first column
      if (g.twiddle && g.log_m > 0) {
        const long long p = (i0 + col) & ((1LL << g.log_m) - 1);
        const int log_lm = g.log_m + LOGL;
        apply_geometric<16>(x, twiddle<DIR>(p * lane, log_lm, T()),
                            twiddle<DIR>(p * 32, log_lm, T()));
      }
      fft512_warp<DIR>(x, lane);  // x[c] = output row (lane >> 1) + 16 c + 256 (lane & 1)
      if constexpr (DIR > 0) {
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) x[c2] = c_scale(x[c2], (T)(1.0 / L));
      }
      const int v0 = (lane >> 1) + 256 * (lane & 1);
      if (g.log_m == 0) {
        // Column col staged contiguously at col * RS, one bulk copy each.
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) cur[col * Cfg::RS + v0 + 16 * c2] = x[c2];
        fence_async_smem();
        __syncthreads();
        if (tid < C) {
          V *dst = out_linear + b * (1LL << g.log_n) + (i0 + tid) * L;
          bulk_store(dst, cur + tid * Cfg::RS, (uint32_t)(L * sizeof(V)));
          bulk_commit();
        }
      } else {
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2)
          *reinterpret_cast<V *>(cb + swz64(((v0 + 16 * c2) << 6) + (col << 3))) = x[c2];
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
          const long long m = 1LL << g.log_m;
          const long long q = i0 >> g.log_m;
          const long long p0 = i0 & (m - 1);
#pragma unroll
          for (int kb = 0; kb < Cfg::BOXES; ++kb)
            tma_store_4d(&tout, cur + kb * Cfg::ROWS_PER_BOX * C, (int)(2 * p0),
                         kb * Cfg::ROWS_PER_BOX, (int)q, (int)b);
          bulk_commit();
        }
      }
      continue;
    }

    const long long b = tile >> g.log_tpb;
    const long long i = (tile & (g.tiles_per_batch - 1)) * C + c;
    // Read even when the wait ran out (the values are then stale but the
    // addresses are the tile's own): the barrier below also carries the
    // verdict.
    V x[P::E];
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = cur[(t + w * P::TP) * C + c];
    // The tile is in registers; buffer s becomes the exchange space.
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicExch(status, kDeviceErrorTimeout);
        // Let the loads issued ahead land before the block exits.
#pragma unroll
        for (int j = 1; j < NB; ++j)
          if (tile + (long long)j * gridDim.x < g.total_tiles)
            mbar_wait(&bar[(k + j) % NB], (uint32_t)((k + j) / NB) & 1u);
      }
      break;
    }
    if (g.twiddle && g.log_m > 0) {
      const long long p = i & ((1LL << g.log_m) - 1);
      const int log_lm = g.log_m + LOGL;
      apply_geometric<P::E>(x, twiddle<DIR>(p * t, log_lm, T()),
                            twiddle<DIR>(p * P::TP, log_lm, T()));
    }

    // No barrier before the first stage's writes: every thread's reads of
    // buffer s happened before the barrier above.
    if constexpr (Cfg::SWIZZLE)
      fft_on_chip<LOGL, DIR, true, false>(x, t, SwzView<V>{cur + c, C}, twt);
    else
      fft_on_chip<LOGL, DIR, true, false>(x, t, SmemView<V>{cur + c, C}, twt);
    if constexpr (DIR > 0) {
#pragma unroll
      for (int w = 0; w < P::E; ++w) x[w] = c_scale(x[w], (T)(1.0 / L));
    }

    __syncthreads();  // the last exchange has been read
    if (g.log_m == 0) {
      // Outputs of butterfly i go to i*L + v: one contiguous block per tile,
      // staged column by column (stride RS) and copied by the bulk-copy
      // engine, one column of L values per thread c < C.
      constexpr int RS = Cfg::RS;
#pragma unroll
      for (int w = 0; w < P::E; ++w) cur[c * RS + t + w * P::TP] = x[w];
      fence_async_smem();
      __syncthreads();
      if (tid < C) {
        V *dst = out_linear + b * (1LL << g.log_n) + ((tile & (g.tiles_per_batch - 1)) * C + tid) * L;
        bulk_store(dst, cur + tid * RS, (uint32_t)(L * sizeof(V)));
        bulk_commit();
      }
    } else {
      // Rows of the output tile are m elements apart: TMA tensor store.
#pragma unroll
      for (int w = 0; w < P::E; ++w) cur[(t + w * P::TP) * C + c] = x[w];
      fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        const long long m = 1LL << g.log_m;
        const long long q = i >> g.log_m;  // same for the whole tile (C <= m)
        const long long p0 = (tile & (g.tiles_per_batch - 1)) * C & (m - 1);
#pragma unroll
        for (int kb = 0; kb < Cfg::BOXES; ++kb)
          tma_store_4d(&tout, cur + kb * Cfg::ROWS_PER_BOX * C, (int)(2 * p0),
                       kb * Cfg::ROWS_PER_BOX, (int)q, (int)b);
        bulk_commit();
      }
    }
  }
  if (tid < C) bulk_wait_all();
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and the persistent launch.
// ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, found through the runtime (no
// link-time dependency on libcuda).
inline EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

inline bool tma_disabled() { return option(FFT_OPT_NO_TMA) == 1; }

// Multiprocessors of the current device (cached per device).
inline int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = cache[dev].load(std::memory_order_acquire);
  if (v == 0 && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
    cache[dev].store(v, std::memory_order_release);
  return v;
}

// Launches the TMA pass kernel, or returns cudaErrorNotSupported (nothing
// launched) when the shape does not suit it: tiles narrower than 2 columns
// (16-byte TMA rows), fewer columns than one tile, output blocks shorter than
// a tile, FFT_OPT_NO_TMA set, or no driver entry point.
template <typename T, int LOGL, int DIR, bool SHFL>
cudaError_t launch_pass_tma_t(const void *in, void *out, int log_n, int log_m, int twiddle,
                              long long batch, cudaStream_t st, int overlap) {
  using Cfg = TmaConfig<T, LOGL, SHFL>;
  if constexpr (!SHFL && TmaConfig<T, LOGL>::SHFL_OK) {
    if (option(FFT_OPT_PASS_SHFL) == 1)
      return launch_pass_tma_t<T, LOGL, DIR, true>(in, out, log_n, log_m, twiddle, batch, st,
                                                   overlap);
  }
  if constexpr (Cfg::C < 2 || LOGL < 4) {
    return cudaErrorNotSupported;
  } else {
    const long long cols = 1LL << (log_n - LOGL);
    EncodeTiledFn enc = encode_tiled();
    const int sms = sm_count();
    // An output tile must not straddle two blocks of length m (C <= m).
    if (tma_disabled() || cols < Cfg::C || (log_m > 0 && (1LL << log_m) < Cfg::C) || !enc ||
        sms <= 0 || batch > 0xffffffffLL)
      return cudaErrorNotSupported;
    const CUtensorMapDataType dt =
        sizeof(T) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT64;
    const cuuint64_t es = sizeof(vec2_t<T>);
    const cuuint64_t n = 1ull << log_n;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    // Input: [batch][L rows][cols] complex, as scalars (re, im) on the
    // innermost axis.
    CUtensorMap tin, tout;
    // The shuffle variant's tiles (64-byte rows) use the 64-byte swizzle.
    const CUtensorMapSwizzle swz = SHFL ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE;
    const cuuint64_t din[3] = {2ull * (cuuint64_t)cols, (cuuint64_t)Cfg::L, (cuuint64_t)batch};
    const cuuint64_t sin_[2] = {(cuuint64_t)cols * es, n * es};
    const cuuint32_t box3[3] = {2u * Cfg::C, (cuuint32_t)Cfg::ROWS_PER_BOX, 1u};
    if (enc(&tin, dt, 3, const_cast<void *>(in), din, sin_, box3, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (log_m > 0) {
      // Output q*L*m + p + v*m: [batch][q][L rows v][m columns p].
      const cuuint64_t m = 1ull << log_m;
      const cuuint64_t Q = n / ((cuuint64_t)Cfg::L * m);
      const cuuint64_t dout[4] = {2ull * m, (cuuint64_t)Cfg::L, Q, (cuuint64_t)batch};
      const cuuint64_t sout[3] = {m * es, (cuuint64_t)Cfg::L * m * es, n * es};
      const cuuint32_t box4[4] = {2u * Cfg::C, (cuuint32_t)Cfg::ROWS_PER_BOX, 1u, 1u};
      if (enc(&tout, dt, 4, out, dout, sout, box4, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    } else {
      tout = tin;  // unused: the first pass stores linearly
    }
    auto kern = fft_pass_tma_kernel<T, LOGL, DIR, SHFL>;
    static DeviceOnce attr_set;
    const cudaError_t attr = smem_limit_once((const void *)kern, Cfg::SMEM, attr_set);
    if (attr != cudaSuccess) return attr;
    TmaGeom g{log_n, log_m, twiddle, cols / Cfg::C, (cols / Cfg::C) * batch, 0, 0,
              log2_pow2(cols / Cfg::C)};
    static std::atomic<int> occupancy[64];
    const int per_sm = blocks_per_sm_once((const void *)kern, Cfg::THREADS, Cfg::SMEM, occupancy);
    long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);
    if (grid > g.total_tiles) grid = g.total_tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tin, tout, static_cast<vec2_t<T> *>(out), g,
                              device_status_word());
  }
}

}  // namespace
}  // namespace fftgb
