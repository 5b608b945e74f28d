// fft_pass_cluster.cuh -- an HBM pass whose on-chip length is split over a
// cluster of R thread blocks that exchange through distributed shared
// memory.
//
// The pass computes what fft_pass.cuh's pass computes (butterfly i reads
// in[i + u*N/L], u < L, multiplies input u by W_{L m}^{p u}, takes the
// L-point DFT and writes out[q*L*m + p + v*m]).  A tile of C columns x L
// rows does not fit one block's shared memory well for L >= 2^11 (64 KB
// and more per block, so few blocks per SM and exposed load latency), so
// the L-point DFT is split in the four-step way ("FFT on GPU", section Fast
// Fourier Transform: a DFT of length R L' as R interleaved DFTs of length
// L', twiddled, then combined by R-point butterflies):
//   u = u1 + R u2 (u1 < R, u2 < L'),  v = v2 + L' v1 (v2 < L', v1 < R),
//   Y[v2 + L' v1] = sum_{u1} W_R^{u1 v1} W_L^{u1 v2} sum_{u2} x[u1 + R u2] W_{L'}^{u2 v2}.
// Block u1 of the cluster loads rows u1, u1 + R, u1 + 2R, ... of the tile
// (one TMA box stream, row stride R*N/L), does the L'-point transforms of
// its C columns on chip and publishes the results in its shared memory.
// After a cluster barrier, block s reads, for its own range of v2 (L'/R of
// them), the R published values of every column from the R blocks
// (ld.shared::cluster), multiplies them by W_L^{u1 v2}, does the R-point
// butterflies, and stores Y[v2 + L' v1] for every v1 from a staging area:
// by TMA tensor store when output rows are m > 1 elements apart, else as
// contiguous runs of L'/R values per column by bulk copies.  A second
// cluster barrier frees the published values for the next tile.
//
// Every block of a cluster walks the same tiles, so all of them reach
// every cluster barrier the same number of times.  The one wait that can
// fail, a block's TMA load (bounded mbarrier wait), is reported to the
// whole cluster: every block writes its status into every block's flag
// array before the first barrier and reads its own array after it, so all
// blocks of the cluster leave together (after one more barrier) and the
// device status word records kDeviceErrorTimeout.
#pragma once

#include "fft_pass_tma.cuh"

namespace fftgb {
namespace {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of all blocks of the cluster: writes before it (shared memory
// included) are visible to reads after it in every block of the cluster.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
// Shared-memory address of the same variable in block `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_cluster(uint32_t addr, float2) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
               : "=f"(v.x), "=f"(v.y)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ double2 ld_cluster(uint32_t addr, double2) {
  double2 v;
  asm volatile("ld.shared::cluster.v2.f64 {%0, %1}, [%2];"
               : "=d"(v.x), "=d"(v.y)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_flag(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// Split of an on-chip length 2^LOGL over a cluster: L' = 2^10 rows per
// block, R = L / L' blocks (2, 4 or 8: L = 2^11 .. 2^13), C columns of 32
// bytes per tile (4 fp32, 2 fp64 complex values).  Shared memory: a load
// buffer (the next tile arrives there while the block works on this one)
// and a work buffer (exchanges of the L'-point transform, then the
// published values, then the staged output); the stage twiddles are
// computed, which leaves room for three blocks per SM.
template <typename T, int LOGL> struct ClusterConfig {
  static constexpr int LOGLP = 10;
  static constexpr bool OK = LOGL > LOGLP && LOGL <= LOGLP + 3;
  static constexpr int R = OK ? 1 << (LOGL - LOGLP) : 1;
  using P = StagePlan<LOGLP>;
  using V = vec2_t<T>;
  static constexpr int L = 1 << LOGL;
  static constexpr int LP = P::L;        // rows each block loads
  static constexpr int LPP = LP / R;     // v2 values each block combines
  static constexpr int C = (int)(32 / sizeof(V));
  static constexpr int THREADS = C * P::TP;
  static constexpr int MIN_BLOCKS = sizeof(T) == 4 ? 3 : 2;  // 80 / 255 registers
  static constexpr int BOX_IN = LP < 256 ? LP : 256;
  // Output boxes (m > 1): 256 rows of C columns.
  static constexpr int BOX_OUT = LPP < 256 ? LPP : 256;
  static constexpr uint32_t TILE_BYTES = (uint32_t)(C * LP * sizeof(V));
  // First-pass staging: column c at c * S1 (S1 = 8 mod 16 spreads the
  // writes of the C lanes that share a row over the banks).
  static constexpr int S1 = LP + 8;
  static constexpr int EXCH = C * P::SMEM_ELEMS;
  static constexpr int STAGE1 = C * S1;
  static constexpr int RAW = EXCH > STAGE1 ? EXCH : STAGE1;
  static constexpr int LOAD_ELEMS = C * LP;
  static constexpr int WORK_ELEMS = ((RAW * (int)sizeof(V) + 127) / 128) * 128 / (int)sizeof(V);
  static constexpr size_t SMEM = 256 + (size_t)(LOAD_ELEMS + WORK_ELEMS) * sizeof(V);
};

template <typename T, int LOGL, int DIR>
__global__ void __launch_bounds__(ClusterConfig<T, LOGL>::THREADS,
                                  ClusterConfig<T, LOGL>::MIN_BLOCKS)
    fft_pass_cluster_kernel(const __grid_constant__ CUtensorMap tin,
                            const __grid_constant__ CUtensorMap tout, vec2_t<T> *out_linear,
                            TmaGeom g, int *status) {
  using Cfg = ClusterConfig<T, LOGL>;
  using P = StagePlan<Cfg::LOGLP>;
  using V = vec2_t<T>;
  constexpr int C = Cfg::C, R = Cfg::R, L = Cfg::L, LP = Cfg::LP, LPP = Cfg::LPP;
  constexpr int KB = 16 / R;  // R-point butterflies per thread
  extern __shared__ __align__(128) unsigned char smem_cl[];
  unsigned char *base = smem_cl + ((128u - (smem_addr(smem_cl) & 127u)) & 127u);
  uint64_t *bar = reinterpret_cast<uint64_t *>(base);
  int *flags = reinterpret_cast<int *>(base + 64);  // [R]: block q's load failed
  V *const lbuf = reinterpret_cast<V *>(base + 128);
  V *const work = lbuf + Cfg::LOAD_ELEMS;

  const int tid = threadIdx.x;
  const int c = tid % C;
  const int t = tid / C;
  const int r = (int)cluster_rank();
  const long long cluster = blockIdx.x / R, nclusters = gridDim.x / R;
  const uint32_t work_addr = smem_addr(work), my_flag = smem_addr(flags + r);

  // Test hook: the failing block arms its first load for 16 bytes and
  // issues no copy (nothing is in flight when it leaves); only its waits
  // are shortened.
  const bool failing = g.debug_fail == r + 1;
  const uint32_t limit = failing && g.poll_limit ? g.poll_limit : 1u << 22;
  auto issue_load = [&](long long tile) {
    const long long b = tile >> g.log_tpb;
    const long long i0 = (tile & (g.tiles_per_batch - 1)) * C;
    mbar_expect_tx(&bar[0], Cfg::TILE_BYTES);
#pragma unroll
    for (int kb = 0; kb < LP / Cfg::BOX_IN; ++kb)
      tma_load_4d(lbuf + kb * Cfg::BOX_IN * C, &tin, &bar[0], (int)(2 * i0), r,
                  kb * Cfg::BOX_IN, (int)b);
  };

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0 && cluster < g.total_tiles) {
    if (failing) mbar_expect_tx(&bar[0], 16);
    else issue_load(cluster);
  }

  int k = 0;
  for (long long tile = cluster; tile < g.total_tiles; tile += nclusters, ++k) {
    const long long b = tile >> g.log_tpb;
    const long long i0 = (tile & (g.tiles_per_batch - 1)) * C;
    const long long next = tile + nclusters;
    const bool ok = mbar_wait(&bar[0], (uint32_t)k & 1u, limit);
    const int bad = __syncthreads_or(!ok);

    // Step 1: rows r + R*(t + w*TP) of column i0 + c, inter-pass twiddle,
    // L'-point transform (x[w] = value v2 = t + w*TP), published.
    V x[P::E];
#pragma unroll
    for (int w = 0; w < P::E; ++w)
      x[w] = bad ? make_c<V>((T)0, (T)0) : lbuf[(t + w * P::TP) * C + c];
    if (tid < C * R) bulk_wait_read_all();  // the previous tile's stores have left `work`
    __syncthreads();  // the load buffer is free; `work` is free
    bool prefetched = false;
    if (tid == 0 && !bad && next < g.total_tiles) {
      issue_load(next);
      prefetched = true;
    }
    if (g.twiddle && g.log_m > 0) {
      const long long p = (i0 + c) & ((1LL << g.log_m) - 1);
      const int log_lm = g.log_m + LOGL;
      apply_geometric<P::E>(x, twiddle<DIR>(p * (r + (long long)R * t), log_lm, T()),
                            twiddle<DIR>(p * R * P::TP, log_lm, T()));
    }
    fft_on_chip<Cfg::LOGLP, DIR>(x, t, SmemView<V>{work + c, C});
    __syncthreads();  // the last exchange has been read
#pragma unroll
    for (int w = 0; w < P::E; ++w) work[(t + w * P::TP) * C + c] = x[w];
    if (tid < R) st_cluster_flag(peer_addr(my_flag, (uint32_t)tid), bad);
    cluster_barrier();  // every block's values and load status are published

    int any_bad = 0;
#pragma unroll
    for (int q = 0; q < R; ++q) any_bad |= flags[q];
    if (any_bad) {
      cluster_barrier();  // no block leaves while another may still read its values
      if (tid == 0) {
        atomicExch(status, kDeviceErrorTimeout);
        // Let the prefetch issued above land before the block exits.
        if (prefetched) mbar_wait(&bar[0], (uint32_t)(k + 1) & 1u, limit);
      }
      break;
    }

    // Step 2: v2 = r*LPP + t + kk*TP; y[kk*R + u1] = published value u1,
    // times W_L^{u1 v2} (powers of W_L^{v2}, at most log2 R products deep).
    V y[P::E];
#pragma unroll
    for (int kk = 0; kk < KB; ++kk) {
      const int v2 = r * LPP + t + kk * P::TP;
      const uint32_t a = work_addr + (uint32_t)((v2 * C + c) * (int)sizeof(V));
#pragma unroll
      for (int q = 0; q < R; ++q) y[kk * R + q] = ld_cluster(peer_addr(a, (uint32_t)q), V());
    }
    cluster_barrier();  // every block has read this block's published values
#pragma unroll
    for (int kk = 0; kk < KB; ++kk) {
      V pw[R];
      powers<R>(twiddle<DIR>((long long)(r * LPP + t + kk * P::TP), LOGL, T()), pw);
#pragma unroll
      for (int q = 1; q < R; ++q) y[kk * R + q] = c_mul(y[kk * R + q], pw[q]);
      dft_reg<R, DIR>(y + kk * R);
    }
    if constexpr (DIR > 0) {
#pragma unroll
      for (int w = 0; w < P::E; ++w) y[w] = c_scale(y[w], (T)(1.0 / L));
    }

    // y[kk*R + v1] is output row v = v1*LP + r*LPP + t + kk*TP of column
    // i0 + c.  Staged in `work`, stored by the bulk-copy engine.
    if (g.log_m == 0) {
      // Outputs of butterfly i go to i*L + v: runs of LPP consecutive
      // values per column and v1, staged as [c][v1*LPP + v2'] and copied
      // run by run.
#pragma unroll
      for (int kk = 0; kk < KB; ++kk)
#pragma unroll
        for (int v1 = 0; v1 < R; ++v1)
          work[c * Cfg::S1 + v1 * LPP + t + kk * P::TP] = y[kk * R + v1];
      fence_async_smem();
      __syncthreads();
      if (tid < C * R) {
        const int cc = tid / R, v1 = tid % R;
        bulk_store(out_linear + (b << g.log_n) + (i0 + cc) * L + v1 * LP + r * LPP,
                   work + cc * Cfg::S1 + v1 * LPP, (uint32_t)(LPP * sizeof(V)));
        bulk_commit();
      }
    } else {
      // Rows m elements apart: staged as [v1][v2'][c].
#pragma unroll
      for (int kk = 0; kk < KB; ++kk)
#pragma unroll
        for (int v1 = 0; v1 < R; ++v1)
          work[(v1 * LPP + t + kk * P::TP) * C + c] = y[kk * R + v1];
      fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        const long long m = 1LL << g.log_m;
        const long long q = i0 >> g.log_m;  // same for the whole tile (C <= m)
        const long long p0 = i0 & (m - 1);
#pragma unroll
        for (int v1 = 0; v1 < R; ++v1)
#pragma unroll
          for (int h = 0; h < LPP / Cfg::BOX_OUT; ++h)
            tma_store_4d(&tout, work + (v1 * LPP + h * Cfg::BOX_OUT) * C, (int)(2 * p0),
                         v1 * LP + r * LPP + h * Cfg::BOX_OUT, (int)q, (int)b);
        bulk_commit();
      }
    }
  }
  if (tid < C * R) bulk_wait_all();
}

inline bool cluster_disabled() { return option(FFT_OPT_NO_CLUSTER) == 1; }

// Shortest on-chip length (log2) that takes the cluster kernel.  Measured
// on GB300 (fp32 2D transforms, column pass on clusters vs one block per
// tile, forward + inverse): 2048^2 x 8 0.511 vs 0.429 ms, 4096^2 x 2 0.534
// vs 0.572 ms, 8192^2 1.31 vs 2.29 ms: columns of 4096 and more.  A 2^26
// transform as two cluster passes of 2^13 (0.85 ms) stays slower than
// three single-block passes of 2^9 (0.61 ms), so the 1D planner keeps its
// short passes.  FFT_OPT_CLUSTER_LOG_MIN (11 .. 13) overrides it for tests.
inline int cluster_min_log() {
  const long long v = option(FFT_OPT_CLUSTER_LOG_MIN);
  return v >= 11 && v <= 13 ? (int)v : 12;
}

// Launches the cluster pass kernel, or returns cudaErrorNotSupported
// (nothing launched) when the shape does not suit it: on-chip length
// outside cluster_min_log() .. 2^13, fewer columns than one tile, output
// blocks shorter than a tile, FFT_OPT_NO_CLUSTER set, no driver entry
// point, or no cluster fits the device.
template <typename T, int LOGL, int DIR>
cudaError_t launch_pass_cluster_t(const void *in, void *out, int log_n, int log_m, int twiddle,
                                  long long batch, cudaStream_t st, int debug_fail,
                                  unsigned poll_limit) {
  using Cfg = ClusterConfig<T, LOGL>;
  if constexpr (!Cfg::OK) {
    return cudaErrorNotSupported;
  } else {
    const long long cols = 1LL << (log_n - LOGL);
    EncodeTiledFn enc = encode_tiled();
    if (cluster_disabled() || LOGL < cluster_min_log() || cols < Cfg::C ||
        (log_m > 0 && (1LL << log_m) < Cfg::C) || !enc || batch > 0xffffffffLL)
      return cudaErrorNotSupported;
    const CUtensorMapDataType dt =
        sizeof(T) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT64;
    const cuuint64_t es = sizeof(vec2_t<T>);
    const cuuint64_t nn = 1ull << log_n;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    // Input row u = u1 + R u2 of column i: [batch][u2 < L'][u1 < R][cols],
    // as scalars on the innermost axis; block u1 loads boxes at u1.
    CUtensorMap tin, tout;
    const cuuint64_t din[4] = {2ull * (cuuint64_t)cols, (cuuint64_t)Cfg::R, (cuuint64_t)Cfg::LP,
                               (cuuint64_t)batch};
    const cuuint64_t sin_[3] = {(cuuint64_t)cols * es, (cuuint64_t)Cfg::R * cols * es, nn * es};
    const cuuint32_t boxi[4] = {2u * Cfg::C, 1u, (cuuint32_t)Cfg::BOX_IN, 1u};
    if (enc(&tin, dt, 4, const_cast<void *>(in), din, sin_, boxi, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (log_m > 0) {
      // Output q*L*m + p + v*m: [batch][q][L rows v][m columns p].
      const cuuint64_t m = 1ull << log_m;
      const cuuint64_t Q = nn / ((cuuint64_t)Cfg::L * m);
      const cuuint64_t dout[4] = {2ull * m, (cuuint64_t)Cfg::L, Q, (cuuint64_t)batch};
      const cuuint64_t sout[3] = {m * es, (cuuint64_t)Cfg::L * m * es, nn * es};
      const cuuint32_t boxo[4] = {2u * Cfg::C, (cuuint32_t)Cfg::BOX_OUT, 1u, 1u};
      if (enc(&tout, dt, 4, out, dout, sout, boxo, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    } else {
      tout = tin;  // unused: the first pass stores contiguous runs
    }
    auto kern = fft_pass_cluster_kernel<T, LOGL, DIR>;
    static DeviceOnce attr_set;
    const cudaError_t attr = smem_limit_once((const void *)kern, Cfg::SMEM, attr_set);
    if (attr != cudaSuccess) return attr;

    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeClusterDimension;
    la[0].val.clusterDim.x = Cfg::R;
    la[0].val.clusterDim.y = 1;
    la[0].val.clusterDim.z = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    // Clusters resident at once (cached per device).
    static std::atomic<int> resident[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
    int ncl = resident[dev].load(std::memory_order_acquire);
    if (ncl == 0) {
      cfg.gridDim = dim3((unsigned)(Cfg::R * sm_count()));
      if (cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg) != cudaSuccess || ncl <= 0) {
        (void)cudaGetLastError();
        return cudaErrorNotSupported;
      }
      resident[dev].store(ncl, std::memory_order_release);
    }
    TmaGeom g{log_n, log_m, twiddle, cols / Cfg::C, (cols / Cfg::C) * batch, debug_fail,
              poll_limit, log2_pow2(cols / Cfg::C)};
    long long clusters = ncl < g.total_tiles ? ncl : g.total_tiles;
    cfg.gridDim = dim3((unsigned)(clusters * Cfg::R));
    return cudaLaunchKernelEx(&cfg, kern, tin, tout, static_cast<vec2_t<T> *>(out), g,
                              device_status_word());
  }
}

}  // namespace
}  // namespace fftgb
