// fft_rows.cuh -- batched contiguous transforms done wholly on chip.
//
// One thread block holds F whole transforms of length N = 2^LOGN
// (N <= 2^14 fp32, 2^13 fp64): each thread loads 16 elements straight from
// HBM (element t + w*N/16, w < 16: a warp reads 32 consecutive elements per
// load), runs every Stockham stage in registers with shared-memory exchanges
// between stages, and writes its 16 results back in the same pattern.  The
// data touches HBM exactly once in each direction ("Stockham FFT Butterfly
// Algorithm in Parallel GLSL", section Performance: batches of butterfly
// steps completed on chip before writing back).
#pragma once

#include "fft_device.cuh"
#include "fft_warp.cuh"
#include "internal.h"

namespace fftgb {
// Kernels and their launchers have internal linkage: every translation unit
// that instantiates one owns its own copy, so no kernel is registered twice.
namespace {

template <typename T, int LOGN> struct RowsConfig {
  using P = StagePlan<LOGN>;
  // Transforms per block: enough to give the block 256 threads.
  static constexpr int F = P::TP >= 256 ? 1 : 256 / P::TP;
  static constexpr int THREADS = P::TP * F;
  static constexpr size_t SMEM = (size_t)F * P::SMEM_ELEMS * sizeof(vec2_t<T>);
};

template <typename T, int LOGN, int DIR>
__global__ void __launch_bounds__(RowsConfig<T, LOGN>::THREADS)
    fft_rows_kernel(const vec2_t<T> *in, vec2_t<T> *out, long long batch) {
  using V = vec2_t<T>;
  using P = StagePlan<LOGN>;
  constexpr int F = RowsConfig<T, LOGN>::F;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V *smem = reinterpret_cast<V *>(smem_raw);

  const int t = threadIdx.x % P::TP;
  const int f = threadIdx.x / P::TP;
  const long long tr = (long long)blockIdx.x * F + f;
  const bool active = tr < batch;

  // Launched with programmatic dependent launch: wait until the previous
  // kernel on the stream has finished (and its writes are visible) before
  // reading, and let the next kernel's blocks be scheduled once every block
  // of this one holds its data (they then fill the SMs this launch's tail
  // frees, and wait the same way).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  V x[P::E];
  if (active) {
    const V *src = in + tr * P::L;
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = src[t + w * P::TP];
  } else {
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = make_c<V>((T)0, (T)0);
  }
  asm volatile("griddepcontrol.launch_dependents;");

  const SmemView<V> sm{smem + f * P::SMEM_ELEMS, 1};
  fft_on_chip<LOGN, DIR, false, false>(x, t, sm);  // data came from global memory

  if (active) {
    V *dst = out + tr * P::L;
#pragma unroll
    for (int w = 0; w < P::E; ++w) {
      V v = x[w];
      if constexpr (DIR > 0) v = c_scale(v, (T)(1.0 / P::L));  // inverse: 1/N
      dst[t + w * P::TP] = v;
    }
  }
}

template <typename T, int LOGN, int DIR>
cudaError_t launch_rows_t(const void *in, void *out, long long batch, cudaStream_t st) {
  using C = RowsConfig<T, LOGN>;
  auto kern = fft_rows_kernel<T, LOGN, DIR>;
  if (C::SMEM > 48 * 1024) {
    static DeviceOnce attr_set;
    const cudaError_t e = smem_limit_once((const void *)kern, C::SMEM, attr_set);
    if (e != cudaSuccess) return e;
  }
  const long long grid = (batch + C::F - 1) / C::F;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
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
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const vec2_t<T> *>(in),
                            static_cast<vec2_t<T> *>(out), batch);
}

// 512-point transforms with the warp-shuffle exchange of fft_warp.cuh: one
// warp per transform, 8 per block, no shared memory (selected by
// FFT_OPT_ROWS_SHFL; the shared-memory engine above is the default).
template <typename T, int DIR>
__global__ void __launch_bounds__(256) fft_rows_warp_kernel(const vec2_t<T> *in, vec2_t<T> *out,
                                                           long long batch) {
  using V = vec2_t<T>;
  const int lane = threadIdx.x & 31;
  const long long tr = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tr >= batch) return;  // whole warps leave together
  asm volatile("griddepcontrol.wait;" ::: "memory");
  V x[16];
  const V *src = in + tr * 512;
#pragma unroll
  for (int r = 0; r < 16; ++r) x[r] = src[lane + 32 * r];
  asm volatile("griddepcontrol.launch_dependents;");
  fft512_warp<DIR>(x, lane);
  V *dst = out + tr * 512 + (lane >> 1) + 256 * (lane & 1);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    V v = x[c];
    if constexpr (DIR > 0) v = c_scale(v, (T)(1.0 / 512));
    dst[16 * c] = v;
  }
}

template <typename T, int DIR>
cudaError_t launch_rows_warp_t(const void *in, void *out, long long batch, cudaStream_t st) {
  const long long grid = (batch + 7) / 8;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fft_rows_warp_kernel<T, DIR>,
                            static_cast<const vec2_t<T> *>(in), static_cast<vec2_t<T> *>(out),
                            batch);
}

template <typename T, int DIR, int LOGN = 0>
cudaError_t dispatch_rows(int logn, const void *in, void *out, long long batch,
                          cudaStream_t st) {
  if constexpr (LOGN > RowsMaxLog<T>::value) {
    return cudaErrorInvalidValue;
  } else {
    if (logn == LOGN) {
      if constexpr (LOGN == 9) {
        if (option(FFT_OPT_ROWS_SHFL) == 1) return launch_rows_warp_t<T, DIR>(in, out, batch, st);
      }
      return launch_rows_t<T, LOGN, DIR>(in, out, batch, st);
    }
    return dispatch_rows<T, DIR, LOGN + 1>(logn, in, out, batch, st);
  }
}

}  // namespace
}  // namespace fftgb
