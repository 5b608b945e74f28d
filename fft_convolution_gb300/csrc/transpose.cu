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

// Tile k of the launch: batch b, first row r0, first column c0.  32-bit
// index arithmetic (the callers check that tile counts and sides fit).
struct TileIndex {
  unsigned b, r0, c0;
  __device__ __forceinline__ TileIndex(unsigned k, unsigned per, unsigned tiles_c) {
    b = k / per;
    const unsigned rem = k - b * per;
    const unsigned tr = rem / tiles_c;
    r0 = tr * kTile;
    c0 = (rem - tr * tiles_c) * kTile;
  }
};

// in [B][R][C] -> out [B][C][R], 32 x 32 tiles through shared memory (one
// spare column: the column reads of 8- and 16-byte elements fall on distinct
// banks).  Blocks loop over the tiles; each thread loads its four elements
// of a tile before storing any.
template <typename V>
__global__ void __launch_bounds__(kTile *kRowsPerPass)
    transpose_kernel(const V *__restrict__ in, V *__restrict__ out, unsigned R, unsigned C,
                     unsigned tiles_r, unsigned tiles_c, unsigned total) {
  __shared__ V tile[kTile][kTile + 1];
  const unsigned per = tiles_r * tiles_c;
  const unsigned tx = threadIdx.x, ty = threadIdx.y;
  for (unsigned k = blockIdx.x; k < total; k += gridDim.x) {
    const TileIndex ti(k, per, tiles_c);
    const size_t base = (size_t)ti.b * R * C;
    const V *src = in + base;
    V *dst = out + base;
    const unsigned c = ti.c0 + tx;
#pragma unroll
    for (int j = 0; j < kTile / kRowsPerPass; ++j) {
      const unsigned r = ti.r0 + ty + j * kRowsPerPass;
      if (r < R && c < C) tile[ty + j * kRowsPerPass][tx] = src[(size_t)r * C + c];
    }
    __syncthreads();
    const unsigned r = ti.r0 + tx;
#pragma unroll
    for (int j = 0; j < kTile / kRowsPerPass; ++j) {
      const unsigned cc = ti.c0 + ty + j * kRowsPerPass;
      if (cc < C && r < R) dst[(size_t)cc * R + r] = tile[tx][ty + j * kRowsPerPass];
    }
    __syncthreads();  // the tile is free for the next one
  }
}

// The same transpose with out[b][c][r] = in[b][r][c] * W_N^{(r c) mod N},
// W_N^e = hi[e >> log_s] * lo[e & (2^log_s - 1)] (the four-step twiddle;
// conjugated for the inverse, conj != 0).
template <typename V>
__global__ void __launch_bounds__(kTile *kRowsPerPass)
    transpose_twiddle_kernel(const V *__restrict__ in, V *__restrict__ out, unsigned R,
                             unsigned C, unsigned tiles_r, unsigned tiles_c, unsigned total,
                             long long N, const V *__restrict__ lo, const V *__restrict__ hi,
                             int log_s, int conj) {
  __shared__ V tile[kTile][kTile + 1];
  const unsigned per = tiles_r * tiles_c;
  const unsigned long long mask = (1ull << log_s) - 1;
  const unsigned tx = threadIdx.x, ty = threadIdx.y;
  for (unsigned k = blockIdx.x; k < total; k += gridDim.x) {
    const TileIndex ti(k, per, tiles_c);
    const size_t base = (size_t)ti.b * R * C;
    const V *src = in + base;
    V *dst = out + base;
    const unsigned c = ti.c0 + tx;
#pragma unroll
    for (int j = 0; j < kTile / kRowsPerPass; ++j) {
      const unsigned r = ti.r0 + ty + j * kRowsPerPass;
      if (r < R && c < C) {
        unsigned long long e = (unsigned long long)r * c;  // < N when R C = N (the four-step)
        if (e >= (unsigned long long)N) e %= (unsigned long long)N;
        V w = c_mul(hi[e >> log_s], lo[e & mask]);
        if (conj) w.y = -w.y;
        tile[ty + j * kRowsPerPass][tx] = c_mul(src[(size_t)r * C + c], w);
      }
    }
    __syncthreads();
    const unsigned r = ti.r0 + tx;
#pragma unroll
    for (int j = 0; j < kTile / kRowsPerPass; ++j) {
      const unsigned cc = ti.c0 + ty + j * kRowsPerPass;
      if (cc < C && r < R) dst[(size_t)cc * R + r] = tile[tx][ty + j * kRowsPerPass];
    }
    __syncthreads();
  }
}

// Tile counts of a [B][R][C] transpose, or false when they do not fit the
// kernels' 32-bit tile arithmetic.
inline bool transpose_tiles(long long B, long long R, long long C, unsigned *tr, unsigned *tc,
                            unsigned *total) {
  const long long r = (R + kTile - 1) / kTile, c = (C + kTile - 1) / kTile;
  if (R >= (1LL << 31) || C >= (1LL << 31) || B * r * c >= (1LL << 31)) return false;
  *tr = (unsigned)r;
  *tc = (unsigned)c;
  *total = (unsigned)(B * r * c);
  return true;
}

template <typename V>
cudaError_t transpose_twiddle_t(const void *in, void *out, long long B, long long R, long long C,
                                long long N, const void *lo, const void *hi, int log_s, int conj,
                                cudaStream_t st) {
  if (B <= 0 || R <= 0 || C <= 0 || N <= 0) return cudaErrorInvalidValue;
  unsigned tr, tc, total;
  if (!transpose_tiles(B, R, C, &tr, &tc, &total)) return cudaErrorInvalidValue;
  const unsigned grid = total < 152u * 16u ? total : 152u * 16u;
  transpose_twiddle_kernel<V><<<grid, dim3(kTile, kRowsPerPass), 0, st>>>(
      static_cast<const V *>(in), static_cast<V *>(out), (unsigned)R, (unsigned)C, tr, tc, total,
      N, static_cast<const V *>(lo), static_cast<const V *>(hi), log_s, conj);
  return cudaGetLastError();
}

template <typename V>
cudaError_t transpose_t(const void *in, void *out, long long B, long long R, long long C,
                        cudaStream_t st) {
  if (B <= 0 || R <= 0 || C <= 0) return cudaErrorInvalidValue;
  unsigned tr, tc, total;
  if (!transpose_tiles(B, R, C, &tr, &tc, &total)) return cudaErrorInvalidValue;
  const unsigned grid = total < 152u * 16u ? total : 152u * 16u;
  transpose_kernel<V><<<grid, dim3(kTile, kRowsPerPass), 0, st>>>(
      static_cast<const V *>(in), static_cast<V *>(out), (unsigned)R, (unsigned)C, tr, tc,
      total);
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
