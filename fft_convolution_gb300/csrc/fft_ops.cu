// fft_ops.cu -- the C ABI's other operations: polynomial products,
// convolutions (device and host buffers), the test hooks, the device status
// word and the status strings.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "plan.h"

using namespace fftgb;

extern "C" {

int polymul_batched(const int64_t *a, int64_t na, const int64_t *b, int64_t nb, int64_t *c,
                    int64_t batch, void *stream) {
  if (!a || !b || !c || na <= 0 || nb <= 0 || batch <= 0) return FFT_ERR_INVALID_ARG;
  if (((uintptr_t)a & 7u) || ((uintptr_t)b & 7u) || ((uintptr_t)c & 7u))
    return FFT_ERR_MISALIGNED;
  const int64_t nc = na + nb - 1;
  const int log_len = nc > 4 ? ilog2_exact(nc) : 2;  // at least a 4-point transform
  if (log_len > 27 || batch > ((int64_t)1 << 36) / ((int64_t)1 << log_len))
    return FFT_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = polymul_scratch_bytes(batch, log_len);
  void *scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, bytes, st);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_polymul(reinterpret_cast<const long long *>(a), na,
                     reinterpret_cast<const long long *>(b), nb, reinterpret_cast<long long *>(c),
                     batch, log_len, scratch, st);
  cudaError_t f = cudaFreeAsync(scratch, st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (f != cudaSuccess) return cuda_fail(f);
  return FFT_OK;
}

int polymul_num_kernels(int64_t na, int64_t nb) {
  if (na <= 0 || nb <= 0) return 0;
  const int64_t nc = na + nb - 1;
  const int log_len = nc > 4 ? ilog2_exact(nc) : 2;
  if (log_len > 27) return 0;
  return fftgb::polymul_num_kernels(log_len);
}

int polymul(const int64_t *a, int64_t na, const int64_t *b, int64_t nb, int64_t *c,
            void *stream) {
  return polymul_batched(a, na, b, nb, c, 1, stream);
}

// Maps the public (kind, h_per_row) to the internal variant and checks the
// lengths; returns FFT_OK and the transform length, or an error.
static int convolve_setup(int64_t nx, int64_t nh, int64_t batch, int h_per_row, int kind,
                          int dtype, int *ikind, int *log_len) {
  if (nx <= 0 || nh <= 0 || batch <= 0 || (h_per_row != 0 && h_per_row != 1) ||
      (kind != FFT_CONV_COMPLEX && kind != FFT_CONV_REAL) ||
      (dtype != FFT_C2C_F32 && dtype != FFT_C2C_F64))
    return FFT_ERR_INVALID_ARG;
  const int64_t ny = nx + nh - 1;
  const int l = ny > 2 ? ilog2_exact(ny) : 1;
  const int max_log = dtype == FFT_C2C_F32 ? 27 : 26;
  if (l > max_log || batch > ((int64_t)1 << 40) / ((int64_t)1 << l)) return FFT_ERR_UNSUPPORTED;
  *ikind = kind == FFT_CONV_COMPLEX ? 0 : (h_per_row ? 2 : 1);
  *log_len = l;
  return FFT_OK;
}

int fft_convolve(const void *x, int64_t nx, const void *h, int64_t nh, void *y, int64_t batch,
                 int h_per_row, int kind, int dtype, void *stream) {
  if (!x || !h || !y) return FFT_ERR_INVALID_ARG;
  int ikind = 0, log_len = 0;
  const int rc = convolve_setup(nx, nh, batch, h_per_row, kind, dtype, &ikind, &log_len);
  if (rc != FFT_OK) return rc;
  const uintptr_t align = (kind == FFT_CONV_COMPLEX ? 8u : 4u) * (dtype == FFT_C2C_F32 ? 1u : 2u);
  if (((uintptr_t)x | (uintptr_t)h | (uintptr_t)y) & (align - 1)) return FFT_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void *scratch = nullptr;
  cudaError_t e = cudaMallocAsync(
      &scratch, convolve_scratch_bytes(batch, h_per_row, ikind, dtype, log_len), st);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_convolve(x, nx, h, nh, y, batch, h_per_row, ikind, dtype, log_len, scratch, st);
  cudaError_t f = cudaFreeAsync(scratch, st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (f != cudaSuccess) return cuda_fail(f);
  return FFT_OK;
}

int fft_convolve_num_kernels(int64_t nx, int64_t nh, int64_t batch, int h_per_row, int kind,
                             int dtype) {
  int ikind = 0, log_len = 0;
  if (convolve_setup(nx, nh, batch, h_per_row, kind, dtype, &ikind, &log_len) != FFT_OK)
    return 0;
  return convolve_num_kernels(ikind, dtype, log_len);
}

int polymul_batched_host(const int64_t *a_host, int64_t na, const int64_t *b_host, int64_t nb,
                         int64_t *c_host, int64_t batch, int64_t *dev_a, int64_t *dev_b,
                         int64_t *dev_c, int64_t chunk, void *stream) {
  if (!a_host || !b_host || !c_host || !dev_a || !dev_b || !dev_c || na <= 0 || nb <= 0 ||
      batch <= 0 || chunk <= 0)
    return FFT_ERR_INVALID_ARG;
  if (((uintptr_t)dev_a & 7u) || ((uintptr_t)dev_b & 7u) || ((uintptr_t)dev_c & 7u))
    return FFT_ERR_MISALIGNED;
  if (polymul_num_kernels(na, nb) == 0) return FFT_ERR_UNSUPPORTED;
  const int64_t nc = na + nb - 1;
  return host_pipeline(
      batch, chunk, static_cast<cudaStream_t>(stream),
      [&](long long b0, long long cnt, cudaStream_t s) {
        cudaError_t e = cudaMemcpyAsync(dev_a + b0 * na, a_host + b0 * na, (size_t)cnt * na * 8,
                                        cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return e;
        return cudaMemcpyAsync(dev_b + b0 * nb, b_host + b0 * nb, (size_t)cnt * nb * 8,
                               cudaMemcpyHostToDevice, s);
      },
      [&](long long b0, long long cnt, cudaStream_t s) {
        const int rc = polymul_batched(dev_a + b0 * na, na, dev_b + b0 * nb, nb, dev_c + b0 * nc,
                                       cnt, s);
        return rc == FFT_OK ? cudaSuccess : (g_cuda_error != cudaSuccess ? g_cuda_error
                                                                          : cudaErrorInvalidValue);
      },
      [&](long long b0, long long cnt, cudaStream_t s) {
        return cudaMemcpyAsync(c_host + b0 * nc, dev_c + b0 * nc, (size_t)cnt * nc * 8,
                               cudaMemcpyDeviceToHost, s);
      });
}

int fft_convolve_host(const void *x_host, int64_t nx, const void *h, int64_t nh, void *y_host,
                      int64_t batch, int h_per_row, int kind, int dtype, void *dev_x, void *dev_y,
                      int64_t chunk, void *stream) {
  if (!x_host || !h || !y_host || !dev_x || !dev_y || chunk <= 0) return FFT_ERR_INVALID_ARG;
  int ikind = 0, log_len = 0;
  const int rc = convolve_setup(nx, nh, batch, h_per_row, kind, dtype, &ikind, &log_len);
  if (rc != FFT_OK) return rc;
  const size_t elem = (kind == FFT_CONV_COMPLEX ? 8 : 4) * (dtype == FFT_C2C_F32 ? 1 : 2);
  const int64_t ny = nx + nh - 1;
  char *dx = static_cast<char *>(dev_x);
  char *dy = static_cast<char *>(dev_y);
  const char *hh = static_cast<const char *>(h);
  return host_pipeline(
      batch, chunk, static_cast<cudaStream_t>(stream),
      [&](long long b0, long long cnt, cudaStream_t s) {
        return cudaMemcpyAsync(dx + (size_t)b0 * nx * elem,
                               static_cast<const char *>(x_host) + (size_t)b0 * nx * elem,
                               (size_t)cnt * nx * elem, cudaMemcpyHostToDevice, s);
      },
      [&](long long b0, long long cnt, cudaStream_t s) {
        const int r = fft_convolve(dx + (size_t)b0 * nx * elem, nx,
                                   hh + (h_per_row ? (size_t)b0 * nh * elem : 0), nh,
                                   dy + (size_t)b0 * ny * elem, cnt, h_per_row, kind, dtype, s);
        return r == FFT_OK ? cudaSuccess : (g_cuda_error != cudaSuccess ? g_cuda_error
                                                                         : cudaErrorInvalidValue);
      },
      [&](long long b0, long long cnt, cudaStream_t s) {
        return cudaMemcpyAsync(static_cast<char *>(y_host) + (size_t)b0 * ny * elem,
                               dy + (size_t)b0 * ny * elem, (size_t)cnt * ny * elem,
                               cudaMemcpyDeviceToHost, s);
      });
}

int fft_debug_radix2_pass(const void *in, void *out, int64_t n, int64_t half, int dtype,
                          void *stream) {
  if (!in || !out || n <= 0 || half <= 0 || n % (2 * half) != 0 ||
      (dtype != FFT_C2C_F32 && dtype != FFT_C2C_F64))
    return FFT_ERR_INVALID_ARG;
  if (misaligned(in) || misaligned(out)) return FFT_ERR_MISALIGNED;
  cudaError_t e = launch_radix2_pass(dtype, in, out, n, half, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return FFT_OK;
}

int fft_debug_wait_timeout(int64_t polls, void *stream) {
  if (polls <= 0 || polls > ((int64_t)1 << 22)) return FFT_ERR_INVALID_ARG;
  cudaError_t e = launch_wait_timeout(polls, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return FFT_OK;
}

int fft_debug_cluster_timeout(void *data, int64_t polls, void *stream) {
  if (!data || polls <= 0 || polls > ((int64_t)1 << 22)) return FFT_ERR_INVALID_ARG;
  if (misaligned(data)) return FFT_ERR_MISALIGNED;
  cudaError_t e = debug_cluster_timeout_f32(data, (unsigned)polls, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return FFT_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(e);
  return FFT_OK;
}

int fft_device_status(void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  int *word = device_status_word();
  if (!word) return cuda_fail(cudaErrorInvalidDevice);
  int v = 0;
  e = cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e);
    return FFT_ERR_DEVICE_TIMEOUT;
  }
  return FFT_OK;
}

int fft_last_status(void) { return g_status; }

int fft_debug_set_option(int option, int64_t value) {
  if (value < 0) return set_option(option, -1) ? FFT_OK : FFT_ERR_INVALID_ARG;
  bool ok;
  switch (option) {
    case FFT_OPT_PASS_LOG: ok = value >= 4 && value <= kPassMaxLogF32; break;
    case FFT_OPT_PASS_SPLIT: ok = value > 0 && value < (1LL << (4 * kMaxPasses)); break;
    case FFT_OPT_NO_TMA:
    case FFT_OPT_NO_CLUSTER:
    case FFT_OPT_ND_ROWS_T:
    case FFT_OPT_ROWS_SHFL:
    case FFT_OPT_PASS_SHFL: ok = value <= 1; break;
    case FFT_OPT_CLUSTER_LOG_MIN: ok = value >= 11 && value <= 13; break;
    case FFT_OPT_COL_RADIX_LOG: ok = value <= 3; break;
    default: ok = false;
  }
  return ok && set_option(option, value) ? FFT_OK : FFT_ERR_INVALID_ARG;
}

const char *fft_status_string(int status) {
  switch (status) {
    case FFT_OK: return "ok";
    case FFT_ERR_INVALID_ARG: return "invalid argument";
    case FFT_ERR_NOT_POW2: return "not a power of two (no longer returned)";
    case FFT_ERR_UNSUPPORTED: return "unsupported size, type or dimensionality";
    case FFT_ERR_CUDA: return "CUDA error";
    case FFT_ERR_ALLOC: return "device allocation failed";
    case FFT_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FFT_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
    default: return "unknown status";
  }
}

const char *fft_last_cuda_error(void) { return cudaGetErrorString(g_cuda_error); }

}  // extern "C"

