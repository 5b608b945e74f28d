// fft_rows_t.cuh -- on-chip row transforms that store their output
// transposed: one pass of a multi-dimensional transform.
//
// A 2D transform is the 1D transform along each axis in turn ("Stockham FFT
// Butterfly Algorithm in Parallel GLSL", section Multi-Dimensional
// Transforms).  Here every axis is transformed as contiguous rows: the
// input [b][R][L] (R rows of length L per matrix) is read row by row as in
// fft_rows.cuh, transformed on chip, and written as [b][L][R], so the next
// axis becomes the contiguous one.  Two passes bring [H][W] back to [H][W],
// three bring [D][H][W] back to [D][H][W]; every read is a contiguous row.
// A block holds F >= 32 bytes / element-size rows, so each output row
// receives F consecutive values (whole 32-byte sectors): the results are
// staged in shared memory as [L][F + 1] (the spare column spreads the
// writes over the banks) and stored F values at a time.
#pragma once

#include "fft_rows.cuh"

namespace fftgb {
namespace {

template <typename T, int LOGN> struct RowsTConfig {
  using P = StagePlan<LOGN>;
  static constexpr int FMIN = (int)(32 / sizeof(vec2_t<T>));
  static constexpr int F = RowsConfig<T, LOGN>::F > FMIN ? RowsConfig<T, LOGN>::F : FMIN;
  static constexpr int THREADS = P::TP * F;
  static constexpr int FS = F + 1;  // staging row stride
  static constexpr size_t EXCH = (size_t)F * P::SMEM_ELEMS;
  static constexpr size_t STAGE = (size_t)P::L * FS;
  static constexpr size_t SMEM = (EXCH > STAGE ? EXCH : STAGE) * sizeof(vec2_t<T>);
  static constexpr bool OK = THREADS <= 1024 && LOGN >= 4 && SMEM <= 227 * 1024;
};

// rows = all rows of the batch (batch * R); log_r = log2 R.
template <typename T, int LOGN, int DIR>
__global__ void __launch_bounds__(RowsTConfig<T, LOGN>::THREADS)
    fft_rows_t_kernel(const vec2_t<T> *in, vec2_t<T> *out, long long rows, int log_r) {
  using V = vec2_t<T>;
  using P = StagePlan<LOGN>;
  using C = RowsTConfig<T, LOGN>;
  constexpr int F = C::F;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  V *smem = reinterpret_cast<V *>(smem_raw);

  const int t = threadIdx.x % P::TP;
  const int f = threadIdx.x / P::TP;
  const long long row0 = (long long)blockIdx.x * F;
  const bool active = row0 + f < rows;

  // Programmatic dependent launch, as the plain row kernel.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  V x[P::E];
  if (active) {
    const V *src = in + (row0 + f) * P::L;
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = src[t + w * P::TP];
  } else {
#pragma unroll
    for (int w = 0; w < P::E; ++w) x[w] = make_c<V>((T)0, (T)0);
  }
  asm volatile("griddepcontrol.launch_dependents;");

  fft_on_chip<LOGN, DIR, false, false>(x, t, SmemView<V>{smem + f * P::SMEM_ELEMS, 1});

  // Stage as [column][row of the block], then store F rows' values of one
  // column together.
  __syncthreads();  // the exchanges are done with shared memory
#pragma unroll
  for (int w = 0; w < P::E; ++w) smem[(t + w * P::TP) * C::FS + f] = x[w];
  __syncthreads();
  const T scale = DIR > 0 ? (T)(1.0 / P::L) : (T)1;
  const long long R = 1LL << log_r;
  for (int e = threadIdx.x; e < P::L * F; e += C::THREADS) {
    const int c = e / F, g = e % F;  // F is a power of two
    const long long gr = row0 + g;
    if (gr < rows) {
      const long long b = gr >> log_r, r = gr & (R - 1);
      V v = smem[c * C::FS + g];
      if constexpr (DIR > 0) v = c_scale(v, scale);
      out[(b * P::L + c) * R + r] = v;
    }
  }
}

template <typename T, int LOGN, int DIR>
cudaError_t launch_rows_t_t(const void *in, void *out, long long rows, int log_r,
                            cudaStream_t st) {
  using C = RowsTConfig<T, LOGN>;
  if constexpr (!C::OK) {
    return cudaErrorNotSupported;
  } else {
    auto kern = fft_rows_t_kernel<T, LOGN, DIR>;
    if (C::SMEM > 48 * 1024) {
      static DeviceOnce attr_set;
      const cudaError_t e = smem_limit_once((const void *)kern, C::SMEM, attr_set);
      if (e != cudaSuccess) return e;
    }
    const long long grid = (rows + C::F - 1) / C::F;
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
                              static_cast<vec2_t<T> *>(out), rows, log_r);
  }
}

template <typename T, int DIR, int LOGN = 4>
cudaError_t dispatch_rows_t(int logn, const void *in, void *out, long long rows, int log_r,
                            cudaStream_t st) {
  if constexpr (LOGN > RowsMaxLog<T>::value) {
    return cudaErrorNotSupported;
  } else {
    if (logn == LOGN) return launch_rows_t_t<T, LOGN, DIR>(in, out, rows, log_r, st);
    return dispatch_rows_t<T, DIR, LOGN + 1>(logn, in, out, rows, log_r, st);
  }
}

}  // namespace
}  // namespace fftgb
