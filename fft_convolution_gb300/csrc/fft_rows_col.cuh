// fft_rows_col.cuh -- the row pass of a 2D (or 3D) transform with the first
// radix-R stage of the column transform folded in.
//
// A 2D transform of an H x W image is 1D transforms along every row, then
// along every column ("Stockham FFT Butterfly Algorithm in Parallel GLSL",
// section Multi-Dimensional Transforms and Separability).  Long columns
// (H >= 1024) would make the column pass move tiles of narrow 32-byte row
// segments.  Instead the column transform of length H = R * M is split by
// one decimation-in-frequency step (the even/odd split of "FFT on GPU",
// section Fast Fourier Transform, with R parts instead of two): with Y the
// row-transformed image and column output index k = R c + d (c < M, d < R),
//     X[R c + d] = sum_{a<M} W_M^{a c} Z_d[a],
//     Z_d[a]     = W_H^{a d} sum_{j<R} Y[a + M j] W_R^{j d}.
// This kernel computes Z: block (image, a) loads the R rows a + M j, runs
// each row's W-point transform on chip (the engine of fft_rows.cuh), takes
// the R-point DFT across the R rows of every column, multiplies output d by
// W_H^{a d} and writes it to row R a + d.  Seen as an [M][R W] array, column
// d W + k2 of that output holds Z_d[.] of image column k2, so the remaining
// M-point column transforms are the ordinary in-place column pass with
// L = M and stride R W, and its output row c of that column is image row
// R c + d -- the natural order.  The data crosses HBM once here and once in
// the column pass, as before, but the column pass now moves rows of R times
// as many bytes.
//
// Rows a + M j are read and rows R a + d written, so input and output must
// be different arrays.
#pragma once

#include "fft_device.cuh"
#include "internal.h"

namespace fftgb {
namespace {

template <typename T, int LOGW, int LOGR> struct RowsColConfig {
  using P = StagePlan<LOGW>;
  // Four or more rows of whole warps synchronise by named barriers (ids
  // 1 .. R).  Measured on GB300 (fp32, forward + inverse): 8 x 2048^2 with
  // R = 4 0.398 -> 0.392 ms; 32 x 1024^2 with R = 2 0.352 -> 0.383 ms, so
  // two-row blocks keep the block-wide barrier.
  static constexpr bool GROUP_SYNC = P::TP % 32 == 0 && LOGR >= 2 && (1 << LOGR) <= 15;
  static constexpr int R = 1 << LOGR;
  static constexpr int THREADS = R * P::TP;
  static constexpr int SE = P::SMEM_ELEMS > P::L + P::L / 16 ? P::SMEM_ELEMS : P::L + P::L / 16;
  static constexpr size_t SMEM = (size_t)R * SE * sizeof(vec2_t<T>);
  static constexpr int COLS = P::E / R;  // columns per thread in the cross-row step
  // fp32: 1024 resident threads per SM (two 512-thread blocks), registers
  // capped at 64, which the kernel fits without spilling (at 85 registers,
  // one block per SM, the 8 x 2048^2 step took 0.434 ms instead of 0.379).
  // fp64: 512 (128 registers; the 16 values a thread holds take 64).
  static constexpr int RESIDENT = sizeof(T) == 8 ? 512 : 1024;
  static constexpr int MIN_BLOCKS = THREADS >= RESIDENT ? 1 : RESIDENT / THREADS;
};

template <typename T, int LOGW, int LOGR, int DIR>
__global__ void __launch_bounds__(RowsColConfig<T, LOGW, LOGR>::THREADS,
                                  RowsColConfig<T, LOGW, LOGR>::MIN_BLOCKS)
    fft_rows_col_kernel(const vec2_t<T> *in, vec2_t<T> *out, int log_h, long long planes) {
  using V = vec2_t<T>;
  using P = StagePlan<LOGW>;
  using Cfg = RowsColConfig<T, LOGW, LOGR>;
  constexpr int R = Cfg::R;
  constexpr int W = P::L;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V *smem = reinterpret_cast<V *>(smem_raw);

  const int t = threadIdx.x % P::TP;
  const int j = threadIdx.x / P::TP;           // row group: row a + M j
  const long long M = 1LL << (log_h - LOGR);
  const long long plane = (long long)(blockIdx.x >> (log_h - LOGR));
  const long long a = blockIdx.x & (M - 1);
  const long long plane_off = plane << (log_h + LOGW);

  // Launched with programmatic dependent launch (as the row kernel): wait
  // for the previous kernel on the stream before reading.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  V x[P::E];
  {
    const V *src = in + plane_off + (a + M * j) * W;
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = src[t + w * P::TP];
  }
  asm volatile("griddepcontrol.launch_dependents;");

  const SmemView<V> sm{smem + j * Cfg::SE, 1};
  // Each row's transform synchronises only its own TP threads (named
  // barrier 1 + j), so the R rows of a block proceed independently until
  // the cross-row step.  The data came from global memory.
  if constexpr (Cfg::GROUP_SYNC) {
    const GroupSync gsync{1 + j, P::TP};
    fft_on_chip<LOGW, DIR, false, false>(x, t, sm, static_cast<const V *>(nullptr), gsync);
    gsync();  // the row's last on-chip exchange has been read
  } else {
    fft_on_chip<LOGW, DIR, false, false>(x, t, sm);
    __syncthreads();
  }
  // Row j's spectrum into its shared-memory row for the cross-row step.
#pragma unroll
  for (int w = 0; w < P::E; ++w) sm.st(t + w * P::TP, x[w]);
  __syncthreads();  // every row's spectrum is in place

  // W_H^{a d}, d < R (conjugate for the inverse).
  V tw[R];
  powers<R>(twiddle<DIR>(a, log_h, T()), tw);
  // Inverse: this pass carries 1/W (rows) and 1/R (the cross-row DFT); the
  // column pass carries 1/M.
  const T scale = DIR > 0 ? (T)(1.0 / ((double)W * R)) : (T)1;

  V *dst = out + plane_off + (long long)R * a * W;
#pragma unroll
  for (int q = 0; q < Cfg::COLS; ++q) {
    const int col = t + (j * Cfg::COLS + q) * P::TP;
    V y[R];
#pragma unroll
    for (int u = 0; u < R; ++u) y[u] = smem[u * Cfg::SE + pad16(col)];
    dft_reg<R, DIR>(y);
#pragma unroll
    for (int d = 0; d < R; ++d) {
      V v = d == 0 ? y[0] : c_mul(y[d], tw[d]);
      if constexpr (DIR > 0) v = c_scale(v, scale);
      dst[(long long)d * W + col] = v;
    }
  }
  (void)planes;
}

template <typename T, int LOGW, int LOGR, int DIR>
cudaError_t launch_rows_col_t(const void *in, void *out, int log_h, long long planes,
                              cudaStream_t st) {
  using C = RowsColConfig<T, LOGW, LOGR>;
  auto kern = fft_rows_col_kernel<T, LOGW, LOGR, DIR>;
  if (C::SMEM > 48 * 1024) {
    static DeviceOnce attr_set;
    const cudaError_t e = smem_limit_once((const void *)kern, C::SMEM, attr_set);
    if (e != cudaSuccess) return e;
  }
  const long long grid = planes << (log_h - LOGR);
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
                            static_cast<vec2_t<T> *>(out), log_h, planes);
}

// logw in [RowsColMinLog, RowsColMaxLog<T>], logr in [1, 3], R * W / 16 <= 1024 threads.
constexpr int kRowsColMinLog = 8;
template <typename T> struct RowsColMaxLog;
template <> struct RowsColMaxLog<float> { static constexpr int value = 12; };
template <> struct RowsColMaxLog<double> { static constexpr int value = 11; };

template <typename T, int DIR, int LOGW = kRowsColMinLog>
cudaError_t dispatch_rows_col(int logw, int logr, const void *in, void *out, int log_h,
                              long long planes, cudaStream_t st) {
  if constexpr (LOGW > RowsColMaxLog<T>::value) {
    return cudaErrorInvalidValue;
  } else {
    if (logw == LOGW) {
      if (logr == 1) return launch_rows_col_t<T, LOGW, 1, DIR>(in, out, log_h, planes, st);
      if (logr == 2) return launch_rows_col_t<T, LOGW, 2, DIR>(in, out, log_h, planes, st);
      if constexpr ((8 << LOGW) / 16 <= 1024 &&
                    (size_t)8 * (((1 << LOGW) * 17) / 16) * sizeof(vec2_t<T>) <= 200 * 1024) {
        if (logr == 3) return launch_rows_col_t<T, LOGW, 3, DIR>(in, out, log_h, planes, st);
      }
      return cudaErrorInvalidValue;
    }
    return dispatch_rows_col<T, DIR, LOGW + 1>(logw, logr, in, out, log_h, planes, st);
  }
}

}  // namespace
}  // namespace fftgb
