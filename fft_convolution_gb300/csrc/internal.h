// internal.h -- declarations shared between the library's translation units
// (kernel launchers and the C ABI in fft_plan.cu, fft_exec.cu, fft_ops.cu).
// Not installed.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <stddef.h>
#include <stdint.h>

#include "fft_gb300.h"

namespace fftgb {

// Largest transform one thread block holds on chip: 2^14 complex fp32 or
// 2^13 complex fp64 (139 KB of shared memory with padding).
template <typename T> struct RowsMaxLog;
template <> struct RowsMaxLog<float> { static constexpr int value = 14; };
template <> struct RowsMaxLog<double> { static constexpr int value = 13; };

// Unique id of the calling thread's current CUDA context (cuCtxGetId), or 0
// when there is none or the driver does not offer the query.  Set-up cached
// per device (a kernel attribute, the device address of a symbol) is keyed
// on it: after cudaDeviceReset the runtime creates a new context with a new
// id, and that set-up is done again there instead of being taken from the
// destroyed one.
unsigned long long context_id();

// Per-device record of the context a piece of set-up was last done in.
struct DeviceOnce {
  std::atomic<unsigned long long> ctx[64];
};

// Process-wide test / tuning options of fft_debug_set_option (FFT_OPT_*
// in the public header; fft_plan.cu): the current value, -1 for the
// library's own choice.
constexpr int kNumOptions = 10;
long long option(int which);
bool set_option(int which, long long value);

// Sets a kernel's dynamic shared-memory limit once per device and context
// (the attribute belongs to the context).  `done` is the calling launcher's
// own record.
inline cudaError_t smem_limit_once(const void *kern, size_t bytes, DeviceOnce &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long id = context_id();
  if (id != 0 && done.ctx[dev].load(std::memory_order_acquire) == id) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.ctx[dev].store(context_id(), std::memory_order_release);
  return e;
}

// Resident blocks per SM of a kernel on the current device, computed once
// per device into the launcher's own `cache`; 0 if the query fails.
inline int blocks_per_sm_once(const void *kern, int threads, size_t smem,
                              std::atomic<int> (&cache)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = cache[dev].load(std::memory_order_acquire);
  if (v == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, smem) ==
                    cudaSuccess)
    cache[dev].store(v, std::memory_order_release);
  return v;
}

// Batched contiguous transforms of length 2^logn (fft_rows_*.cu).
cudaError_t launch_rows_f32(int logn, int dir, const void *in, void *out, long long batch,
                            cudaStream_t st);
cudaError_t launch_rows_f64(int logn, int dir, const void *in, void *out, long long batch,
                            cudaStream_t st);

// Row pass of 2D / 3D transforms with the first radix-2^logr stage of the
// column transform folded in (rows_col_*.cu): `planes` H x W planes
// (H = 2^log_h, W = 2^logw), out of place; the column pass that follows
// runs with on-chip length H / 2^logr over columns at stride 2^logr W.
// cudaErrorInvalidValue outside rows_col_supported().
cudaError_t launch_rows_col_f32(int logw, int logr, int dir, const void *in, void *out, int log_h,
                                long long planes, cudaStream_t st);
cudaError_t launch_rows_col_f64(int logw, int logr, int dir, const void *in, void *out, int log_h,
                                long long planes, cudaStream_t st);
inline bool rows_col_supported(bool f64, int logw, int logr) {
  if (logw < 8 || logw > (f64 ? 11 : 12) || logr < 1 || logr > 3) return false;
  if ((1 << (logw + logr - 4)) > 1024) return false;  // threads per block
  const long long smem = (1LL << logr) * (((1LL << logw) * 17) / 16) * (f64 ? 16 : 8);
  return logr < 3 || smem <= 200 * 1024;
}

// One pass of a transform that does not fit on chip, or the column pass of
// a 2D transform (fft_pass_*.cu).  The data of each of `batch` transforms is
// 2^log_n elements; the pass does 2^(log_n - log_l) on-chip transforms of
// length 2^log_l, each over the elements i + u * 2^(log_n - log_l),
// u < 2^log_l, and is the radix-2^log_l Stockham stage whose previous block
// length is 2^log_m.  With twiddle != 0 input u of butterfly i is first
// multiplied by W_{2^(log_l+log_m)}^{(i mod 2^log_m) u}.  overlap != 0
// lets the TMA pass kernel start while the previous kernel on the stream
// drains (programmatic dependent launch): set only after another pass,
// whose persistent grid leaves no room for the new blocks until it
// retires -- after a kernel of many short waves the new persistent blocks
// would sit on SM resources that kernel still needs.
struct PassArgs {
  int log_n;
  int log_l;
  int log_m;
  int twiddle;
  long long batch;
  int overlap = 0;
};
cudaError_t launch_pass_f32(int dir, const PassArgs &a, const void *in, void *out,
                            cudaStream_t st);
cudaError_t launch_pass_f64(int dir, const PassArgs &a, const void *in, void *out,
                            cudaStream_t st);
// Largest on-chip length a pass kernel is built for.
constexpr int kPassMaxLogF32 = 14;
constexpr int kPassMaxLogF64 = 13;

// Device status word that bounded in-kernel waits set when they run out
// (fft_plan.cu; fft_device_status reads and clears it).
int *device_status_word();

// Bounded-wait test hook (debug_pass.cu).
cudaError_t launch_wait_timeout(long long polls, cudaStream_t st);
// One cluster pass (2^15 fp32 points in place) whose block 1 waits for a
// load that never completes (fft_pass_f32.cu).
cudaError_t debug_cluster_timeout_f32(void *data, unsigned polls, cudaStream_t st);

// One radix-2 butterfly pass (debug_pass.cu).
cudaError_t launch_radix2_pass(int dtype, const void *in, void *out, long long n, long long half,
                               cudaStream_t st);

// Fused polynomial multiplication (polymul.cu): transforms of length
// 2^log_len (2 <= log_len <= 27) over `batch` pairs; scratch must hold
// polymul_scratch_bytes(batch, log_len) bytes.
size_t polymul_scratch_bytes(long long batch, int log_len);
int polymul_num_kernels(int log_len);
cudaError_t launch_polymul(const long long *a, long long na, const long long *b, long long nb,
                           long long *c, long long batch, int log_len, void *scratch,
                           cudaStream_t st);

// Linear convolution of signals (conv.cu).  kind: 0 complex, 1 real rows in
// pairs (shared real filter), 2 real rows one at a time.
size_t convolve_scratch_bytes(long long batch, int h_per_row, int kind, int dtype, int log_len);
int convolve_num_kernels(int kind, int dtype, int log_len);
int convolve_passes(int dtype, int log_len);  // HBM passes per multi-pass transform
cudaError_t launch_convolve(const void *x, long long nx, const void *h, long long nh, void *y,
                            long long batch, int h_per_row, int kind, int dtype, int log_len,
                            void *scratch, cudaStream_t st);
cudaError_t launch_convolve_f32(const void *x, long long nx, const void *h, long long nh, void *y,
                                long long batch, int h_per_row, int kind, int log_len,
                                void *scratch, cudaStream_t st);
cudaError_t launch_convolve_f64(const void *x, long long nx, const void *h, long long nh, void *y,
                                long long batch, int h_per_row, int kind, int log_len,
                                void *scratch, cudaStream_t st);

// Transforms of any length (anylen_*.cu): direct DFT (N <= 64) and
// Bluestein through a power-of-two convolution of length 2^log_m.
cudaError_t bluestein_prepare_f32(long long N, int log_m, int dir, void *w, void *B, void *ws,
                                  cudaStream_t st);
cudaError_t bluestein_prepare_f64(long long N, int log_m, int dir, void *w, void *B, void *ws,
                                  cudaStream_t st);
cudaError_t bluestein_exec_f32(const void *in, void *out, long long N, long long batch, int log_m,
                               double scale, void *w, void *B, void *ws, cudaStream_t st);
cudaError_t bluestein_exec_f64(const void *in, void *out, long long N, long long batch, int log_m,
                               double scale, void *w, void *B, void *ws, cudaStream_t st);
cudaError_t dft_small_f32(const void *in, void *out, int N, long long batch, int dir, double scale,
                          cudaStream_t st);
cudaError_t dft_small_f64(const void *in, void *out, int N, long long batch, int dir, double scale,
                          cudaStream_t st);

// Mixed-radix on-chip transforms (mixed_*.cu): stage k has radix radix[k]
// (2, 3, 4, 5, 7, 8, 11, 13, 15 or 16) and block length m[k] (the product of the
// radices before it); its forward twiddles W_{R m}^{p u} sit at
// tw_off[k] + (u - 1) m + p of the plan's table.  A block holds F transforms.
struct MixedStages {
  int N;
  int nstages;
  int F;
  int radix[16];
  int m[16];
  int tw_off[16];
  // floor(2^32 / d) + 1 for d = N / radix[k] and d = m[k] (0 when d = 1):
  // floor(x / d) = umulhi(x, magic) while x * d < 2^32.
  unsigned nb_magic[16];
  unsigned m_magic[16];
  // Stages whose butterflies are walked q-fastest (bit k of qorder): the
  // middle stages with odd R and odd m < 16, whose shared-memory stores at
  // q R m + p + v m then run at the odd stride R m across a warp (free of
  // bank conflicts) instead of in runs of m.  nq[k] = N / (R m) and its
  // magic number q_magic[k] split the butterfly index as p * nq + q.
  unsigned qorder;
  int nq[16];
  unsigned q_magic[16];
};
constexpr int kMixedMaxF32 = 12288;  // 2 buffers of N values within 192 KB of shared memory
constexpr int kMixedMaxF64 = 6144;
cudaError_t mixed_exec_f32(const void *in, void *out, long long batch, const MixedStages &ms,
                           const void *tw, int dir, cudaStream_t st);
cudaError_t mixed_exec_f64(const void *in, void *out, long long batch, const MixedStages &ms,
                           const void *tw, int dir, cudaStream_t st);

// Row transforms with transposed stores (rows_t_*.cu): `rows` rows of
// length 2^logn, R = 2^log_r rows per matrix, [b][R][L] in -> [b][L][R] out.
// cudaErrorNotSupported outside 4 <= logn <= rows_t_max_log_*().
cudaError_t launch_rows_t_f32(int logn, int dir, const void *in, void *out, long long rows,
                              int log_r, cudaStream_t st);
cudaError_t launch_rows_t_f64(int logn, int dir, const void *in, void *out, long long rows,
                              int log_r, cudaStream_t st);
int rows_t_max_log_f32();
int rows_t_max_log_f64();

// Batched transpose of complex matrices, in [B][R][C] -> out [B][C][R]
// (transpose.cu); in and out must not overlap.
cudaError_t transpose_complex(int f64, const void *in, void *out, long long B, long long R,
                              long long C, cudaStream_t st);
// The same with out[b][c][r] = in[b][r][c] W_N^{(r c) mod N}, W_N^e from the
// split table hi[e >> log_s] lo[e & (2^log_s - 1)] of the forward root,
// conjugated when conj != 0.
cudaError_t transpose_twiddle_complex(int f64, const void *in, void *out, long long B,
                                      long long R, long long C, long long N, const void *lo,
                                      const void *hi, int log_s, int conj, cudaStream_t st);

// Transforms of real sequences (real_*.cu).  On chip: N = 2H, H = 2^logh,
// forward (dir < 0) batch x 2H reals -> batch x (H + 1) bins, inverse the
// reverse with 1/N.
cudaError_t launch_real_rows_f32(int logh, int dir, const void *in, void *out, long long batch,
                                 cudaStream_t st);
cudaError_t launch_real_rows_f64(int logh, int dir, const void *in, void *out, long long batch,
                                 cudaStream_t st);
// Kernels around a complex plan.  `len` is H for REAL_POST / REAL_PRE and
// the real length N for the others; lo / hi / log_s / nhi describe the
// split twiddle table of W_N (REAL_TABLES fills it).
enum RealAuxOp {
  REAL_TABLES = 0,  // lo[j] = W_N^j (j < 2^log_s), hi[i] = W_N^{i 2^log_s} (i < nhi)
  REAL_POST = 1,    // Z (batch x H) -> X (batch x (H + 1))
  REAL_PRE = 2,     // X (batch x (H + 1)) -> Z (batch x H)
  REAL_WIDEN = 3,   // odd N: reals -> complex with imaginary part 0
  REAL_NARROW = 4,  // odd N: bins 0 .. N/2 of each row
  REAL_EXTEND = 5,  // odd N: half spectrum -> full Hermitian spectrum
  REAL_PART = 6     // odd N: complex -> real parts
};
struct RealAuxArgs {
  const void *in;
  void *out;
  long long len;
  long long batch;
  const void *lo;
  const void *hi;
  int log_s;
  long long nhi;
};
cudaError_t real_aux_f32(int op, const RealAuxArgs &a, cudaStream_t st);
cudaError_t real_aux_f64(int op, const RealAuxArgs &a, cudaStream_t st);

}  // namespace fftgb
