// debug_pass.cu -- one gather-shaped radix-2 butterfly pass, kept as a test
// hook for the single-pass unit check ("The Butterfly: One Thread, One
// Output", gpu.rocks FFT butterfly task 2).  Each thread owns one output
// cell i: j = floor(i/half) mod 2 says whether it is the lower (0) or upper
// (1) member of its pair, base = i - j*half is the lower member's index,
// r = i mod half its position in the half-block; a = in[base],
// b = in[base + half], w = e^{-i pi r / half}; the cell receives a + w b
// (lower) or a - w b (upper).  Nothing is swapped and no thread writes two
// cells.
#include "fft_pass_tma.cuh"

namespace fftgb {

template <typename T>
__global__ void radix2_pass_kernel(const vec2_t<T> *in, vec2_t<T> *out, long long n,
                                   long long half) {
  using V = vec2_t<T>;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const long long j = (i / half) % 2;
  const long long base = i - j * half;
  const long long r = i % half;
  const V a = in[base];
  const V b = in[base + half];
  T s, c;
  if constexpr (sizeof(T) == 4) sincospif((float)r / (float)half, &s, &c);
  else sincospi((double)r / (double)half, &s, &c);
  const V wb = c_mul(make_c<V>(c, -s), b);  // e^{-i pi r/half} * b
  out[i] = (j == 0) ? c_add(a, wb) : c_sub(a, wb);
}

// Test hook for the bounded waits: one block arms an mbarrier with a
// 16-byte transaction that nothing delivers, polls it `polls` times and,
// when the wait runs out, records kDeviceErrorTimeout in the device status
// word -- the same path the TMA pass kernel takes.  No copy is issued, so
// nothing is left in flight when the block exits.
__global__ void wait_timeout_kernel(long long polls, int *status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_expect_tx(&bar, 16);
  }
  __syncthreads();
  bool ok = false;
  for (long long it = 0; it < polls && !ok; ++it) ok = mbar_try_wait(&bar, 0);
  if (__syncthreads_or(!ok) && threadIdx.x == 0) atomicExch(status, kDeviceErrorTimeout);
}

cudaError_t launch_wait_timeout(long long polls, cudaStream_t st) {
  int *status = device_status_word();
  if (!status) return cudaErrorInvalidDevice;
  wait_timeout_kernel<<<1, 32, 0, st>>>(polls, status);
  return cudaGetLastError();
}

cudaError_t launch_radix2_pass(int dtype, const void *in, void *out, long long n, long long half,
                               cudaStream_t st) {
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  if (dtype == 0)
    radix2_pass_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(
        static_cast<const float2 *>(in), static_cast<float2 *>(out), n, half);
  else
    radix2_pass_kernel<double><<<(unsigned)blocks, threads, 0, st>>>(
        static_cast<const double2 *>(in), static_cast<double2 *>(out), n, half);
  return cudaGetLastError();
}

}  // namespace fftgb
