// transpose.cu -- batched transposes of complex matrices, the data movement
// between the axes of a multi-dimensional transform whose sides are not all
// powers of two ("Stockham FFT Butterfly Algorithm in Parallel GLSL",
// section Multi-Dimensional Transforms: the 1D transform along each axis in
// turn; an axis that is not contiguous is brought to the contiguous position
// and back).
#include <cuda_runtime.h>

#include "fft_device.cuh"
#include "internal.h"

namespace fftgb {
namespace {

constexpr int kTile = 32;
constexpr int kRowsPerPass = 8;  // block = 32 x 8 threads

// in [B][R][C] -> out [B][C][R], 32 x 32 tiles through shared memory (one
// spare column: the column reads of 8- and 16-byte elements fall on distinct
// banks).  Blocks loop over the tiles.
template <typename V>
__global__ void __launch_bounds__(kTile *kRowsPerPass)
    transpose_kernel(const V *__restrict__ in, V *__restrict__ out, long long R, long long C,
                     long long tiles_r, long long tiles_c, long long total) {
  __shared__ V tile[kTile][kTile + 1];
  const long long per = tiles_r * tiles_c;
  for (long long k = blockIdx.x; k < total; k += gridDim.x) {
    const long long b = k / per, rem = k - b * per;
    const long long r0 = (rem / tiles_c) * kTile, c0 = (rem % tiles_c) * kTile;
    const V *src = in + b * R * C;
    V *dst = out + b * R * C;
    for (int j = threadIdx.y; j < kTile; j += kRowsPerPass) {
      const long long r = r0 + j, c = c0 + threadIdx.x;
      if (r < R && c < C) tile[j][threadIdx.x] = src[r * C + c];
    }
    __syncthreads();
    for (int j = threadIdx.y; j < kTile; j += kRowsPerPass) {
      const long long c = c0 + j, r = r0 + threadIdx.x;
      if (c < C && r < R) dst[c * R + r] = tile[threadIdx.x][j];
    }
    __syncthreads();  // the tile is free for the next one
  }
}

// The same transpose with out[b][c][r] = in[b][r][c] * W_N^{(r c) mod N},
// W_N^e = hi[e >> log_s] * lo[e & (2^log_s - 1)] (the four-step twiddle;
// conjugated for the inverse, conj != 0).
template <typename V>
__global__ void __launch_bounds__(kTile *kRowsPerPass)
    transpose_twiddle_kernel(const V *__restrict__ in, V *__restrict__ out, long long R,
                             long long C, long long tiles_r, long long tiles_c, long long total,
                             long long N, const V *__restrict__ lo, const V *__restrict__ hi,
                             int log_s, int conj) {
  __shared__ V tile[kTile][kTile + 1];
  const long long per = tiles_r * tiles_c;
  const long long mask = (1LL << log_s) - 1;
  for (long long k = blockIdx.x; k < total; k += gridDim.x) {
    const long long b = k / per, rem = k - b * per;
    const long long r0 = (rem / tiles_c) * kTile, c0 = (rem % tiles_c) * kTile;
    const V *src = in + b * R * C;
    V *dst = out + b * R * C;
    for (int j = threadIdx.y; j < kTile; j += kRowsPerPass) {
      const long long r = r0 + j, c = c0 + threadIdx.x;
      if (r < R && c < C) {
        long long e = r * c;  // < N when R C = N (the four-step), so no reduction
        if (e >= N) e %= N;
        V w = c_mul(hi[e >> log_s], lo[e & mask]);
        if (conj) w.y = -w.y;
        tile[j][threadIdx.x] = c_mul(src[r * C + c], w);
      }
    }
    __syncthreads();
    for (int j = threadIdx.y; j < kTile; j += kRowsPerPass) {
      const long long c = c0 + j, r = r0 + threadIdx.x;
      if (c < C && r < R) dst[c * R + r] = tile[threadIdx.x][j];
    }
    __syncthreads();
  }
}

template <typename V>
cudaError_t transpose_twiddle_t(const void *in, void *out, long long B, long long R, long long C,
                                long long N, const void *lo, const void *hi, int log_s, int conj,
                                cudaStream_t st) {
  if (B <= 0 || R <= 0 || C <= 0 || N <= 0) return cudaErrorInvalidValue;
  const long long tr = (R + kTile - 1) / kTile, tc = (C + kTile - 1) / kTile;
  const long long total = B * tr * tc;
  long long grid = total < 152LL * 16 ? total : 152LL * 16;
  transpose_twiddle_kernel<V><<<(unsigned)grid, dim3(kTile, kRowsPerPass), 0, st>>>(
      static_cast<const V *>(in), static_cast<V *>(out), R, C, tr, tc, total, N,
      static_cast<const V *>(lo), static_cast<const V *>(hi), log_s, conj);
  return cudaGetLastError();
}

template <typename V>
cudaError_t transpose_t(const void *in, void *out, long long B, long long R, long long C,
                        cudaStream_t st) {
  if (B <= 0 || R <= 0 || C <= 0) return cudaErrorInvalidValue;
  const long long tr = (R + kTile - 1) / kTile, tc = (C + kTile - 1) / kTile;
  const long long total = B * tr * tc;
  long long grid = total < 152LL * 16 ? total : 152LL * 16;
  transpose_kernel<V><<<(unsigned)grid, dim3(kTile, kRowsPerPass), 0, st>>>(
      static_cast<const V *>(in), static_cast<V *>(out), R, C, tr, tc, total);
  return cudaGetLastError();
}

}  // namespace

cudaError_t transpose_twiddle_complex(int f64, const void *in, void *out, long long B,
                                      long long R, long long C, long long N, const void *lo,
                                      const void *hi, int log_s, int conj, cudaStream_t st) {
  return f64 ? transpose_twiddle_t<double2>(in, out, B, R, C, N, lo, hi, log_s, conj, st)
             : transpose_twiddle_t<float2>(in, out, B, R, C, N, lo, hi, log_s, conj, st);
}

cudaError_t transpose_complex(int f64, const void *in, void *out, long long B, long long R,
                              long long C, cudaStream_t st) {
  return f64 ? transpose_t<double2>(in, out, B, R, C, st)
             : transpose_t<float2>(in, out, B, R, C, st);
}

}  // namespace fftgb
