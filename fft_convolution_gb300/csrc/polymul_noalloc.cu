// polymul_noalloc.cu -- polynomial multiplication that allocates no device
// memory.
//
// polymul() takes its fp64 scratch from the stream-ordered allocator.  Some
// callers cannot do that at the point where they need a product: a plug-in
// running inside a host application that owns the whole device-memory budget
// and does not let its guests allocate, or a latency-critical loop in which
// an allocation may wait on the device or fail under memory pressure.  This
// entry point gives them the same product with its scratch in a fixed array
// that is part of the library's device image: every GPU that loads the
// library holds those 3 MiB until the process exits, and no call allocates
// or frees anything.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  Nothing in it needs to start at zero: every transform
// pass writes each element it hands to the next pass, and the zero padding
// of the inputs is produced by the first pass's loads, not read from the
// scratch.  Calls whose work overlaps on the GPU (different streams, or
// different host threads without ordering) race on the array and give wrong
// results; order them on one stream or serialise them.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/fft_gb300.h"
#include "internal.h"

namespace {

constexpr long long kMaxLen = FFT_POLYMUL_NOALLOC_MAX_LEN;  // largest transform length L

// 3 MiB of fp64 complex scratch: room for the transforms of one product of
// length up to kMaxLen.  In host code this name is only a stand-in for the
// device array: its device address comes from cudaGetSymbolAddress below,
// once per device.
static __device__ __align__(256) double2 g_noalloc_scratch[3 * kMaxLen];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_on_device[kMaxDevices];
unsigned long long g_scratch_context[kMaxDevices];  // context the address belongs to

int ilog2_ceil(long long n) {
  int l = 0;
  while ((1LL << l) < n) ++l;
  return l;
}

}  // namespace

extern "C" int polymul_noalloc(const int64_t *a, int64_t na, const int64_t *b, int64_t nb,
                               int64_t *c, void *stream) {
  if (!a || !b || !c || na <= 0 || nb <= 0) return FFT_ERR_INVALID_ARG;
  if (((uintptr_t)a & 7u) || ((uintptr_t)b & 7u) || ((uintptr_t)c & 7u))
    return FFT_ERR_MISALIGNED;
  const long long nc = (long long)na + (long long)nb - 1;
  const int log_len = nc > 4 ? ilog2_ceil(nc) : 2;
  if ((1LL << log_len) > kMaxLen ||
      fftgb::polymul_scratch_bytes(1, log_len) > sizeof(g_noalloc_scratch))
    return FFT_ERR_UNSUPPORTED;  // beyond the fixed scratch

  // Set-up, once per device (and again if the device's context was
  // destroyed by cudaDeviceReset and created anew), with that device
  // current: the device address of the scratch array.
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return FFT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FFT_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    const unsigned long long ctx = fftgb::context_id();
    if (!g_scratch_on_device[dev] || ctx == 0 || g_scratch_context[dev] != ctx) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p) return FFT_ERR_CUDA;
      g_scratch_on_device[dev] = p;
      g_scratch_context[dev] = fftgb::context_id();
    }
    scratch = g_scratch_on_device[dev];
  }

  e = fftgb::launch_polymul(reinterpret_cast<const long long *>(a), na,
                            reinterpret_cast<const long long *>(b), nb,
                            reinterpret_cast<long long *>(c), /*batch=*/1, log_len, scratch,
                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FFT_OK : FFT_ERR_CUDA;
}
