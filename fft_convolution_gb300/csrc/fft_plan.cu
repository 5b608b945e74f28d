// fft_plan.cu -- plans: argument checks, the choice of kernels for every
// kind of transform, and the plan's device memory (fft_plan_create,
// fft_plan_create_nd, fft_plan_destroy, fft_plan_workspace_bytes of the C ABI
// in include/fft_gb300.h).
//
// The pages' own boundary is `solve(signal, spectrum, N)` on interleaved
// fp32 device buffers ("FFT on GPU", section FFT on GPU), which launches one
// kernel per butterfly stage with a device-wide synchronisation after each.
// Here a plan fixes the kernel sequence once; fft_exec (fft_exec.cu) only
// enqueues it on the caller's stream and never synchronises.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>
#include <utility>

#include "plan.h"

using namespace fftgb;

// Device status word of the bounded in-kernel waits (0 = no error).
static __device__ int g_device_status;

namespace fftgb {

thread_local int g_status = FFT_OK;
thread_local cudaError_t g_cuda_error = cudaSuccess;

unsigned long long context_id() {
  // cuCtxGetCurrent / cuCtxGetId from the driver, found through the runtime
  // (no link-time dependency on libcuda).
  using GetCurrentFn = CUresult (*)(CUcontext *);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
  static const std::pair<GetCurrentFn, GetIdFn> fns = [] {
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    const bool ok =
        cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess;
    return ok ? std::make_pair(reinterpret_cast<GetCurrentFn>(a), reinterpret_cast<GetIdFn>(b))
              : std::make_pair(static_cast<GetCurrentFn>(nullptr), static_cast<GetIdFn>(nullptr));
  }();
  if (!fns.first) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (fns.first(&ctx) != CUDA_SUCCESS || !ctx || fns.second(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// The device address of g_device_status, looked up once per device and
// context (cudaGetSymbolAddress) and cached.
int *device_status_word() {
  static std::mutex mu;
  static unsigned long long ctx_of[64];
  static int *word_of[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  const unsigned long long id = context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (id == 0 || ctx_of[dev] != id || !word_of[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    word_of[dev] = static_cast<int *>(p);
    ctx_of[dev] = context_id();
  }
  return word_of[dev];
}

// Records a failed CUDA call and consumes the runtime's last-error state it
// left (a failed allocation would otherwise surface again at the next
// launch check of an unrelated call).
int cuda_fail(cudaError_t e) {
  g_cuda_error = e;
  (void)cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? FFT_ERR_ALLOC : FFT_ERR_CUDA;
}

// Process-wide test / tuning options (fft_debug_set_option); -1 = the
// library's own choice.
static std::atomic<long long> g_options[kNumOptions] = {
    {-1}, {-1}, {-1}, {-1}, {-1}, {-1}, {-1}, {-1}, {-1}, {-1}};

long long option(int which) {
  return which > 0 && which < kNumOptions ? g_options[which].load(std::memory_order_relaxed) : -1;
}

bool set_option(int which, long long value) {
  if (which <= 0 || which >= kNumOptions) return false;
  g_options[which].store(value < 0 ? -1 : value, std::memory_order_relaxed);
  return true;
}

// Largest on-chip factor (log2) per HBM pass of a long 1D transform.  The
// default 9 keeps every pass tile at 64 KB with 16 (fp32) / 8 (fp64)
// contiguous columns (FFT_OPT_PASS_LOG overrides it).
int pass_log_limit(int dtype) {
  const long long v = option(FFT_OPT_PASS_LOG);
  const int lim = v >= 4 ? (int)v : 9;
  const int hard = dtype == FFT_C2C_F32 ? kPassMaxLogF32 : kPassMaxLogF64;
  return lim > hard ? hard : lim;
}

// FFT_OPT_PASS_SPLIT: the passes of a multi-pass transform of 2^logn
// points, first pass first (4 bits each), when the factors add up to logn
// and each is within 1 .. the pass kernels' limit.  Returns the number of
// passes, or 0 (no override, or one that does not apply).
static int pass_split_override(int logn, int dtype, int *split) {
  long long v = option(FFT_OPT_PASS_SPLIT);
  if (v <= 0) return 0;
  const int hard = dtype == FFT_C2C_F32 ? kPassMaxLogF32 : kPassMaxLogF64;
  int count = 0, sum = 0;
  while (v > 0) {
    const int f = (int)(v & 15);
    v >>= 4;
    if (f < 1 || f > hard || count == kMaxPasses) return 0;
    split[count++] = f;
    sum += f;
  }
  return count >= 2 && sum == logn ? count : 0;
}

}  // namespace fftgb


extern "C" void fft_plan_destroy(fft_plan *plan);

// Plans `batch` transforms of real sequences of length n (the caller
// validated the arguments; cdtype is the complex type of the samples'
// precision).  N = 2H with H a power of two that fits on chip: one kernel per
// direction.  Other even N: a complex plan of length H and a pre/post
// kernel with a split twiddle table of W_N (computed here on the legacy
// default stream, waited for).  Odd N: a complex plan of length N.
static fft_plan *plan_real(int64_t n, int64_t batch, int direction, int cdtype) {
  const size_t elem = cdtype == FFT_C2C_F32 ? 8 : 16;
  const int on_chip_max = cdtype == FFT_C2C_F32 ? RowsMaxLog<float>::value : RowsMaxLog<double>::value;
  fft_plan *p = new (std::nothrow) fft_plan;
  if (!p) {
    g_status = FFT_ERR_ALLOC;
    return nullptr;
  }
  memset(p, 0, sizeof(*p));
  p->n = n;
  p->batch = batch;
  p->elems = n;
  p->rank = 1;
  p->dims = 1;
  p->direction = direction;
  p->dtype = cdtype;
  p->real = 1;
  if (n % 2 == 0 && is_pow2(n) && ilog2_exact(n) - 1 <= on_chip_max) {
    p->kind = KIND_REAL_ROWS;
    p->logn = ilog2_exact(n) - 1;
    return p;
  }
  const bool even = n % 2 == 0;
  const int64_t inner_n = even ? n / 2 : n;
  p->kind = even ? KIND_REAL_EVEN : KIND_REAL_ODD;
  p->inner = fft_plan_create(inner_n, batch, 1, direction, cdtype);
  if (!p->inner) {  // g_status says why
    delete p;
    return nullptr;
  }
  g_status = FFT_OK;
  p->ws_stride = (size_t)inner_n * elem;
  p->workspace_bytes = (size_t)batch * p->ws_stride;
  cudaError_t e = cudaMalloc(&p->workspace, p->workspace_bytes);
  if (e == cudaSuccess && even) {
    const int64_t H = n / 2;
    int log_s = 0;
    while (((int64_t)1 << (2 * log_s)) < H + 1) ++log_s;
    p->rtw_log_s = log_s;
    p->rtw_nhi = (H >> log_s) + 1;
    p->aux_bytes = (((size_t)1 << log_s) + (size_t)p->rtw_nhi) * elem;
    e = cudaMalloc(&p->rtw, p->aux_bytes);
    if (e == cudaSuccess) {
      char *lo = static_cast<char *>(p->rtw);
      RealAuxArgs a{nullptr, nullptr, n, 0, lo, lo + ((size_t)1 << log_s) * elem, log_s, p->rtw_nhi};
      e = real_aux(cdtype, REAL_TABLES, a, 0);
      if (e == cudaSuccess) e = cudaStreamSynchronize(0);
    }
  }
  if (e != cudaSuccess) {
    g_cuda_error = e;
    (void)cudaGetLastError();
    fft_plan_destroy(p);
    g_status = e == cudaErrorMemoryAllocation ? FFT_ERR_ALLOC : FFT_ERR_CUDA;
    return nullptr;
  }
  return p;
}

// The stages of a mixed-radix plan of length n: the odd factors first (a 3
// and a 5 together as radix 15 while both remain, then 3s, 5s, 7s, 11s, 13s:
// short blocks m while the stride N/R is odd), then the power of two as
// radix-16 stages.  The power of two left over (2, 4 or 8 = 4 * 2) joins
// remaining odd primes as prime-factor radices -- 4 with a 5 or a 3 (20,
// 12), 2 with a 5, a 3 or a 7 (10, 6, 14) -- placed after the odd stages,
// one stage fewer per pairing; what finds no partner stays one 2, 4 or 8
// stage.  False if n has a prime factor above 13 or needs more than 16
// stages.
static bool mixed_stages(int64_t n, int elem, MixedStages *ms) {
  int odd[64], no = 0, a = 0;
  int64_t r = n;
  while (r % 2 == 0) {
    r /= 2;
    ++a;
  }
  // A 3 and a 5 merge into one radix-15 stage (an in-register prime-factor
  // DFT: one shared-memory round trip fewer), first.
  while (r % 15 == 0 && no < 64) {
    r /= 15;
    odd[no++] = 15;
  }
  const int primes[5] = {3, 5, 7, 11, 13};
  for (int f : primes)
    while (r % f == 0 && no < 64) {
      r /= f;
      odd[no++] = f;
    }
  if (r != 1) return false;
  int rest2[2], nr = 0;
  if (a % 4 == 3) {
    rest2[nr++] = 4;
    rest2[nr++] = 2;
  } else if (a % 4) {
    rest2[nr++] = 1 << (a % 4);
  }
  int pfa[2], np = 0, single2 = 1;
  for (int i = 0; i < nr; ++i) {
    const int q = rest2[i];
    const int partners[3] = {5, 3, 7};
    int at = -1;
    for (int w = 0; w < 3 && at < 0; ++w) {
      if (partners[w] == 7 && q != 2) continue;  // 28 values: too many registers
      for (int j = 0; j < no; ++j)
        if (odd[j] == partners[w]) {
          at = j;
          break;
        }
    }
    if (at >= 0) {
      pfa[np++] = q * odd[at];
      odd[at] = 0;
    } else {
      single2 *= q;
    }
  }
  int radix[64], k = 0;
  for (int j = 0; j < no && k < 64; ++j)
    if (odd[j]) radix[k++] = odd[j];
  for (int j = 0; j < np && k < 64; ++j) radix[k++] = pfa[j];
  if (single2 > 1 && k < 64) radix[k++] = single2;
  for (int j = 0; j < a / 4 && k < 64; ++j) radix[k++] = 16;
  if (k > 16) return false;
  // The last stage writes global memory in runs of m = N / R consecutive
  // values.  When a prime-factor last stage writes runs shorter than 16
  // values and moving the largest radix to the front lengthens them to 16
  // or more, do so.  Measured (fp32, forward + inverse of 131072
  // transforms, ms): 100 = 5 * 20 0.121, as 20 * 5 0.095; 96 = 6 * 16
  // 0.107, as 16 * 6 0.144 (so a power-of-two last stage stays).
  if (k >= 2 && n / radix[k - 1] < 16 && (radix[k - 1] & (radix[k - 1] - 1)) != 0) {
    int big = 0;
    for (int j = 1; j < k; ++j)
      if (radix[j] > radix[big]) big = j;
    const int last = big == k - 1 ? radix[k - 2] : radix[k - 1];
    if (big != 0 && n / last >= 16) {
      const int rb = radix[big];
      for (int j = big; j > 0; --j) radix[j] = radix[j - 1];
      radix[0] = rb;
    }
  }
  memset(ms, 0, sizeof(*ms));
  ms->N = (int)n;
  ms->nstages = k;
  auto magic = [](int64_t d) -> unsigned {
    return d > 1 ? (unsigned)(((uint64_t)1 << 32) / (uint64_t)d + 1) : 0u;
  };
  int m = 1, off = 0;
  for (int j = 0; j < k; ++j) {
    ms->radix[j] = radix[j];
    ms->m[j] = m;
    ms->tw_off[j] = off;
    ms->nb_magic[j] = magic(n / radix[j]);
    ms->m_magic[j] = magic(m);
    ms->nq[j] = (int)(n / ((int64_t)radix[j] * m));
    ms->q_magic[j] = magic(ms->nq[j]);
    if (j > 0 && j + 1 < k && m > 1 && m < 16 && (m & 1) && (radix[j] & 1))
      ms->qorder |= 1u << j;
    off += (radix[j] - 1) * m;
    m *= radix[j];
  }
  // Transforms per block: about 2048 values, both buffers within 48 KB.
  int F = n < 2048 ? (int)(2048 / n) : 1;
  while (F > 1 && 2 * (size_t)F * n * elem > 48 * 1024) --F;
  ms->F = F;
  return true;
}

// Forward twiddles of every mixed-radix stage, W_{R m}^{p u} at
// tw_off + (u - 1) m + p, computed in double precision with the exponent
// reduced mod R m, rounded once to the element type.
static void mixed_twiddles(const MixedStages &ms, bool f64, void *host) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int k = 0; k < ms.nstages; ++k) {
    const int R = ms.radix[k], m = ms.m[k];
    const int64_t RM = (int64_t)R * m;
    for (int u = 1; u < R; ++u)
      for (int p = 0; p < m; ++p) {
        const int64_t e = ((int64_t)p * u) % RM;
        const double ang = two_pi * (double)e / (double)RM;
        const size_t at = (size_t)ms.tw_off[k] + (size_t)(u - 1) * m + p;
        if (f64) {
          static_cast<double *>(host)[2 * at] = cos(ang);
          static_cast<double *>(host)[2 * at + 1] = -sin(ang);
        } else {
          static_cast<float *>(host)[2 * at] = (float)cos(ang);
          static_cast<float *>(host)[2 * at + 1] = (float)-sin(ang);
        }
      }
  }
}

// True when every prime factor of n is at most 13 (the mixed-radix kernel's
// radices).
static bool is_smooth_13(int64_t n) {
  const int f[6] = {2, 3, 5, 7, 11, 13};
  for (int k = 0; k < 6; ++k)
    while (n % f[k] == 0) n /= f[k];
  return n == 1;
}

// Split twiddle table of W_N = e^{-2 pi i / N}: lo[j] = W_N^j (j < 2^log_s),
// hi[i] = W_N^{i 2^log_s} (i < nhi), host double precision, rounded once.
static void split_twiddles(int64_t n, int log_s, int64_t nhi, bool f64, void *host) {
  const double two_pi = 6.283185307179586476925286766559;
  const int64_t S = (int64_t)1 << log_s;
  for (int64_t i = 0; i < S + nhi; ++i) {
    const int64_t e = i < S ? i % n : (int64_t)(((unsigned __int128)(i - S) * (unsigned __int128)S) % (unsigned __int128)n);
    const double ang = two_pi * (double)e / (double)n;
    if (f64) {
      static_cast<double *>(host)[2 * i] = cos(ang);
      static_cast<double *>(host)[2 * i + 1] = -sin(ang);
    } else {
      static_cast<float *>(host)[2 * i] = (float)cos(ang);
      static_cast<float *>(host)[2 * i + 1] = (float)-sin(ang);
    }
  }
}

// Four-step plan of a smooth length n = n1 * n2 (p: the caller's plan,
// already holding n, batch, direction, dtype; freed on failure).  x viewed
// as [n1][n2]: transpose, n2 * batch transforms of length n1, twiddle
// W_N^{n2 k1} folded into the second transpose, n1 * batch transforms of
// length n2, transpose to the output order k1 + n1 k2.
static fft_plan *plan_four_step(int64_t n, int64_t n1, int64_t batch, int direction, int dtype,
                                fft_plan *p) {
  const size_t elem = dtype == FFT_C2C_F32 ? 8 : 16;
  const int64_t n2 = n / n1;
  p->kind = KIND_FOUR_STEP;
  p->side[0] = n1;
  p->side[1] = n2;
  cudaError_t e = cudaSuccess;
  p->axis_plan[0] = fft_plan_create(n1, batch * n2, 1, direction, dtype);
  if (p->axis_plan[0]) p->axis_plan[1] = fft_plan_create(n2, batch * n1, 1, direction, dtype);
  if (!p->axis_plan[0] || !p->axis_plan[1]) {
    const int st = g_status;
    fft_plan_destroy(p);
    g_status = st;
    return nullptr;
  }
  g_status = FFT_OK;
  int log_s = 0;
  while (((int64_t)1 << (2 * log_s)) < n) ++log_s;
  p->rtw_log_s = log_s;
  p->rtw_nhi = ((n - 1) >> log_s) + 1;
  p->aux_bytes = (((size_t)1 << log_s) + (size_t)p->rtw_nhi) * elem;
  void *host = malloc(p->aux_bytes);
  e = host ? cudaMalloc(&p->rtw, p->aux_bytes) : cudaErrorMemoryAllocation;
  if (e == cudaSuccess) {
    split_twiddles(n, log_s, p->rtw_nhi, dtype == FFT_C2C_F64, host);
    e = cudaMemcpy(p->rtw, host, p->aux_bytes, cudaMemcpyHostToDevice);
  }
  free(host);
  if (e == cudaSuccess) {
    p->ws_stride = (size_t)n * elem;
    p->workspace_bytes = (size_t)batch * p->ws_stride;
    e = cudaMalloc(&p->workspace, p->workspace_bytes);
    if (e != cudaSuccess) p->workspace = nullptr;
  }
  if (e != cudaSuccess) {
    g_cuda_error = e;
    (void)cudaGetLastError();
    fft_plan_destroy(p);
    g_status = e == cudaErrorMemoryAllocation ? FFT_ERR_ALLOC : FFT_ERR_CUDA;
    return nullptr;
  }
  return p;
}

// Plans a 1D length that is not a power of two (the caller validated the
// other arguments): the direct DFT for n <= kDirectDftMax; mixed radix on
// chip for longer lengths whose prime factors are 2, 3, 5, 7, 11, 13 (up to
// kMixedMaxF32 / kMixedMaxF64); Bluestein for the rest, whose chirp and
// filter spectrum are computed here (on the legacy default stream, waited
// for before returning).
static fft_plan *plan_any_length(int64_t n, int64_t batch, int direction, int dtype) {
  const size_t elem = dtype == FFT_C2C_F32 ? 8 : 16;
  const int on_chip_max = dtype == FFT_C2C_F32 ? RowsMaxLog<float>::value : RowsMaxLog<double>::value;
  fft_plan *p = new (std::nothrow) fft_plan;
  if (!p) {
    g_status = FFT_ERR_ALLOC;
    return nullptr;
  }
  memset(p, 0, sizeof(*p));
  p->n = n;
  p->batch = batch;
  p->elems = n;
  p->rank = 1;
  p->dims = 1;
  p->direction = direction;
  p->dtype = dtype;
  if (n <= kDirectDftMax) {
    p->kind = KIND_DFT;
    return p;
  }
  if (n <= (dtype == FFT_C2C_F32 ? kMixedMaxF32 : kMixedMaxF64) &&
      mixed_stages(n, (int)elem, &p->ms)) {
    p->kind = KIND_MIXED;
    const MixedStages &ms = p->ms;
    const int last = ms.nstages - 1;
    const size_t entries = (size_t)ms.tw_off[last] + (size_t)(ms.radix[last] - 1) * ms.m[last];
    p->aux_bytes = (entries > 0 ? entries : 1) * elem;
    void *host = malloc(p->aux_bytes);
    cudaError_t e = host ? cudaMalloc(&p->mtw, p->aux_bytes) : cudaErrorMemoryAllocation;
    if (e == cudaSuccess) {
      mixed_twiddles(ms, dtype == FFT_C2C_F64, host);
      e = cudaMemcpy(p->mtw, host, entries * elem, cudaMemcpyHostToDevice);
    }
    free(host);
    if (e != cudaSuccess) {
      g_cuda_error = e;
      (void)cudaGetLastError();
      if (p->mtw) cudaFree(p->mtw);
      delete p;
      g_status = e == cudaErrorMemoryAllocation ? FFT_ERR_ALLOC : FFT_ERR_CUDA;
      return nullptr;
    }
    return p;
  }
  const int64_t mixed_max = dtype == FFT_C2C_F32 ? kMixedMaxF32 : kMixedMaxF64;
  if (n > mixed_max && is_smooth_13(n)) {
    // Smooth but longer than one block: the four-step split N = N1 N2 with
    // both factors on chip, N1 the divisor closest to sqrt(N).
    int64_t n1 = 0;
    for (int64_t d = 1; d * d <= n; ++d)
      if (n % d == 0 && n / d <= mixed_max) n1 = d;
    if (n1 > 1 && batch <= ((int64_t)1 << 40) / n) return plan_four_step(n, n1, batch, direction, dtype, p);
  }
  const int log_m = ilog2_exact(2 * n - 1);
  if (log_m > (dtype == FFT_C2C_F32 ? 27 : 26) || batch > ((int64_t)1 << 40) / ((int64_t)1 << log_m)) {
    delete p;
    g_status = FFT_ERR_UNSUPPORTED;
    return nullptr;
  }
  p->kind = KIND_BLUESTEIN;
  p->log_m = log_m;
  const size_t M = (size_t)1 << log_m;
  const size_t chirp_bytes = (((size_t)n * elem + 255) / 256) * 256;
  p->aux_bytes = chirp_bytes + M * elem;
  cudaError_t e = cudaMalloc(&p->chirp, p->aux_bytes);
  if (e == cudaSuccess && log_m > on_chip_max) {
    p->workspace_bytes = 2 * (size_t)batch * M * elem;
    e = cudaMalloc(&p->workspace, p->workspace_bytes);
  }
  if (e == cudaSuccess) {
    p->filter = static_cast<char *>(p->chirp) + chirp_bytes;
    e = dtype == FFT_C2C_F32
            ? bluestein_prepare_f32(n, log_m, direction, p->chirp, p->filter, p->workspace, 0)
            : bluestein_prepare_f64(n, log_m, direction, p->chirp, p->filter, p->workspace, 0);
    if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  }
  if (e != cudaSuccess) {
    g_cuda_error = e;
    (void)cudaGetLastError();
    if (p->workspace) cudaFree(p->workspace);
    if (p->chirp) cudaFree(p->chirp);
    delete p;
    g_status = e == cudaErrorMemoryAllocation ? FFT_ERR_ALLOC : FFT_ERR_CUDA;
    return nullptr;
  }
  return p;
}

// Whether a power-of-two 2D / 3D plan runs every axis as rows with
// transposed stores instead of rows plus column passes.  Measured on GB300
// (fp32, one forward transform): faster when every side is 128 or 256
// (256^2 x 512: 0.163 vs 0.170 ms; 128x256x256 x 4: 0.253 vs 0.264;
// 256^3 x 2: 0.249 vs 0.264), slower for longer sides (2048^2 x 8: 0.240 vs
// 0.209; 512^2 x 128: 0.188 vs 0.175; 32x512^2 x 4: 0.306 vs 0.263) and for
// shorter ones (64^3 x 256: 0.649 vs 0.540).  FFT_OPT_ND_ROWS_T = 0 / 1
// forces the choice (sides 2^4 .. the transposed-store limit) for tuning.
static int nd_rows_t_wanted(int rank, const int *logs, int dtype) {
  const int lim = dtype == FFT_C2C_F32 ? rows_t_max_log_f32() : rows_t_max_log_f64();
  int ok = 1, preferred = 1;
  for (int k = 0; k < rank; ++k) {
    if (logs[k] < 4 || logs[k] > lim) ok = 0;
    if (logs[k] < 7 || logs[k] > 8) preferred = 0;
  }
  const long long forced = option(FFT_OPT_ND_ROWS_T);
  if (forced >= 0) return ok && forced != 0;
  return ok && preferred;
}

// Plans a 2D / 3D transform whose sides are not all powers of two within
// the one-kernel-per-axis limits (the caller validated the arguments and
// the sizes).  The contiguous axis runs as a 1D plan of any length over
// batch * (other sides) rows.  Every other axis of length > 1 runs as an
// in-place power-of-two column pass when its length and its stride are
// powers of two within the pass limits; otherwise it is transposed to the
// contiguous position in the workspace, transformed there by a 1D plan of
// any length, and transposed back.
static fft_plan *plan_nd_any(int rank, const int64_t *shape, int64_t batch, int direction,
                             int dtype) {
  const size_t elem = dtype == FFT_C2C_F32 ? 8 : 16;
  const int pass_max = dtype == FFT_C2C_F32 ? kPassMaxLogF32 : kPassMaxLogF64;
  fft_plan *p = new (std::nothrow) fft_plan;
  if (!p) {
    g_status = FFT_ERR_ALLOC;
    return nullptr;
  }
  memset(p, 0, sizeof(*p));
  p->kind = KIND_ND_ANY;
  p->rank = rank;
  p->dims = rank;
  p->batch = batch;
  p->direction = direction;
  p->dtype = dtype;
  int64_t total = 1;
  for (int k = 0; k < rank; ++k) {
    p->side[k] = shape[k];
    total *= shape[k];
  }
  p->elems = total;
  p->n = shape[rank - 1];
  bool need_ws = false;
  int64_t stride = 1;  // product of the sides inside axis k
  for (int k = rank - 1; k >= 0; --k) {
    const int64_t L = shape[k];
    if (L > 1) {
      const bool pow2_pass = k < rank - 1 && is_pow2(L) && is_pow2(stride) &&
                             ilog2_exact(L) <= pass_max;
      if (pow2_pass) {
        p->axis_pass[k] = 1;
      } else {
        p->axis_plan[k] = fft_plan_create(L, batch * (total / L), 1, direction, dtype);
        if (!p->axis_plan[k]) {  // g_status says why
          const int st = g_status;
          fft_plan_destroy(p);
          g_status = st;
          return nullptr;
        }
        if (k < rank - 1) need_ws = true;
      }
    }
    stride *= L;
  }
  g_status = FFT_OK;
  if (need_ws) {
    p->ws_stride = (size_t)total * elem;
    p->workspace_bytes = (size_t)batch * p->ws_stride;
    cudaError_t e = cudaMalloc(&p->workspace, p->workspace_bytes);
    if (e != cudaSuccess) {
      g_cuda_error = e;
      (void)cudaGetLastError();
      p->workspace = nullptr;
      fft_plan_destroy(p);
      g_status = e == cudaErrorMemoryAllocation ? FFT_ERR_ALLOC : FFT_ERR_CUDA;
      return nullptr;
    }
  }
  return p;
}

extern "C" {

fft_plan *fft_plan_create(int64_t n, int64_t batch, int dims, int direction, int dtype) {
  g_status = FFT_OK;
  if (dims == 2) {
    if (dtype == FFT_REAL_F32 || dtype == FFT_REAL_F64) {
      g_status = FFT_ERR_UNSUPPORTED;  // real transforms are 1D
      return nullptr;
    }
    const int64_t shape[2] = {n, n};
    return fft_plan_create_nd(2, shape, batch, direction, dtype);
  }
  const bool real = dtype == FFT_REAL_F32 || dtype == FFT_REAL_F64;
  if (n <= 0 || batch <= 0 || dims != 1 || (direction != FFT_FORWARD && direction != FFT_INVERSE) ||
      (dtype != FFT_C2C_F32 && dtype != FFT_C2C_F64 && !real)) {
    g_status = FFT_ERR_INVALID_ARG;
    return nullptr;
  }
  if (real) return plan_real(n, batch, direction, dtype == FFT_REAL_F32 ? FFT_C2C_F32 : FFT_C2C_F64);
  if (!is_pow2(n)) return plan_any_length(n, batch, direction, dtype);
  const int logn = ilog2_exact(n);
  const int on_chip_max = dtype == FFT_C2C_F32 ? RowsMaxLog<float>::value : RowsMaxLog<double>::value;
  const size_t elem = dtype == FFT_C2C_F32 ? 8 : 16;

  fft_plan *p = new (std::nothrow) fft_plan;
  if (!p) {
    g_status = FFT_ERR_ALLOC;
    return nullptr;
  }
  memset(p, 0, sizeof(*p));
  p->n = n;
  p->batch = batch;
  p->elems = n;
  p->rank = 1;
  p->dims = 1;
  p->direction = direction;
  p->dtype = dtype;
  p->logn = logn;

  if (logn <= on_chip_max) {
    p->kind = KIND_ROWS;
    return p;
  }
  const int max_log_1d = dtype == FFT_C2C_F32 ? 30 : 29;
  if (logn > max_log_1d || batch > ((int64_t)1 << 40) / n) {
    delete p;
    g_status = FFT_ERR_UNSUPPORTED;
    return nullptr;
  }
  // Stockham passes over HBM: logn split into nearly equal factors of at
  // most pass_log_limit bits, larger factors first (or the split
  // FFT_OPT_PASS_SPLIT names).
  int split[kMaxPasses];
  int P = pass_split_override(logn, dtype, split);
  if (P == 0) {
    const int lim = pass_log_limit(dtype);
    P = (logn + lim - 1) / lim;
    if (P < 2) P = 2;
    if (P > kMaxPasses) {
      delete p;
      g_status = FFT_ERR_UNSUPPORTED;
      return nullptr;
    }
    for (int k = 0; k < P; ++k) split[k] = logn / P + (k < logn % P ? 1 : 0);
  }
  p->kind = KIND_MULTI;
  p->npasses = P;
  for (int k = 0; k < P; ++k) p->pass_log[k] = split[k];
  p->workspace_bytes = (size_t)batch * (size_t)n * elem;
  cudaError_t e = cudaMalloc(&p->workspace, p->workspace_bytes);
  if (e != cudaSuccess) {
    g_cuda_error = e;
    (void)cudaGetLastError();
    delete p;
    g_status = FFT_ERR_ALLOC;
    return nullptr;
  }
  return p;
}

fft_plan *fft_plan_create_nd(int rank, const int64_t *shape, int64_t batch, int direction,
                             int dtype) {
  g_status = FFT_OK;
  if (rank == 1 && shape) return fft_plan_create(shape[0], batch, 1, direction, dtype);
  if ((rank != 2 && rank != 3) || !shape || batch <= 0 ||
      (direction != FFT_FORWARD && direction != FFT_INVERSE) ||
      (dtype != FFT_C2C_F32 && dtype != FFT_C2C_F64)) {
    g_status = FFT_ERR_INVALID_ARG;
    return nullptr;
  }
  const int on_chip_max = dtype == FFT_C2C_F32 ? RowsMaxLog<float>::value : RowsMaxLog<double>::value;
  const int pass_max = dtype == FFT_C2C_F32 ? kPassMaxLogF32 : kPassMaxLogF64;
  int logs[3] = {0, 0, 0};
  int total_log = 0;
  bool fast = true;  // every side a power of two within the one-kernel-per-axis limits
  int64_t total = 1;
  for (int k = 0; k < rank; ++k) {
    if (shape[k] <= 0 || shape[k] > ((int64_t)1 << 30)) {
      g_status = shape[k] <= 0 ? FFT_ERR_INVALID_ARG : FFT_ERR_UNSUPPORTED;
      return nullptr;
    }
    total *= shape[k];
    if (total > ((int64_t)1 << 40)) {
      g_status = FFT_ERR_UNSUPPORTED;
      return nullptr;
    }
    if (!is_pow2(shape[k])) {
      fast = false;
      continue;
    }
    logs[k] = ilog2_exact(shape[k]);
    total_log += logs[k];
    // The innermost side runs on chip; the others as in-place column passes.
    if (logs[k] > (k == rank - 1 ? on_chip_max : pass_max)) fast = false;
  }
  if (batch > ((int64_t)1 << 40) / total) {
    g_status = FFT_ERR_UNSUPPORTED;
    return nullptr;
  }
  if (!fast) return plan_nd_any(rank, shape, batch, direction, dtype);
  fft_plan *p = new (std::nothrow) fft_plan;
  if (!p) {
    g_status = FFT_ERR_ALLOC;
    return nullptr;
  }
  memset(p, 0, sizeof(*p));
  p->kind = KIND_ND;
  p->rank = rank;
  p->dims = rank;
  for (int k = 0; k < rank; ++k) p->shape_log[k] = logs[k];
  // Every axis as on-chip rows with transposed stores (contiguous reads in
  // every pass) when each side fits one such block.
  p->nd_rows_t = nd_rows_t_wanted(rank, logs, dtype);
  p->n = shape[rank - 1];
  p->logn = logs[rank - 1];
  p->elems = (int64_t)1 << total_log;
  p->batch = batch;
  p->direction = direction;
  p->dtype = dtype;
  // Columns of 1024 to 8192 points: fold the first radix-R stage of the
  // column transform into the row pass so that the column pass transforms
  // columns R times shorter of R times wider rows (out-of-place execution
  // only).  1024 and 2048 points take R = 2 and 4 (512-point column
  // passes) where the row pass keeps blocks of at most 512 threads; 4096
  // and 8192 points take R = 4 (1024- and 2048-point column passes instead
  // of cluster passes) where that holds, else R = 2.  Measured on GB300
  // (fp32, forward + inverse, ms): 1024^2 x 32 0.404 unfolded, 0.366 R = 2,
  // 0.382 R = 4; 2048^2 x 8 0.427 unfolded, 0.441 R = 2, 0.420 R = 4, 0.503
  // R = 8 (and 0.444 with R = 4 split over a cluster of two 256-thread
  // blocks); 4096 x 256 x 16 0.264 unfolded, 0.214 R = 2, 0.208 R = 4;
  // 4096 x 1024 x 4 0.270, 0.224, 0.215; 4096^2 x 2 0.527, 0.458, 0.486;
  // 8192 x 1024 x 2 0.295, 0.271, 0.226; 8192 x 2048 0.292, 0.271, 0.231;
  // fp64 8192 x 512 x 2 3.15, 3.11, 2.89.
  if (!p->nd_rows_t) {
    const int logh = logs[rank - 2], logw = logs[rank - 1];
    const long long forced = option(FFT_OPT_COL_RADIX_LOG);
    int logr = 0;
    if (forced >= 0) logr = (int)forced;
    else if ((logh == 10 || logh == 11) && logw >= 4 && (logh - 9) + logw - 4 <= 9) logr = logh - 9;
    else if (logh == 12 || logh == 13) logr = 2 + logw - 4 <= 9 ? 2 : 1;
    if (logr >= 1 && logr < logh && rows_col_supported(dtype == FFT_C2C_F64, logw, logr))
      p->col_radix_log = logr;
  }
  if (p->nd_rows_t) {
    p->ws_stride = (size_t)p->elems * (dtype == FFT_C2C_F32 ? 8 : 16);
    p->workspace_bytes = (size_t)batch * p->ws_stride;
    cudaError_t e = cudaMalloc(&p->workspace, p->workspace_bytes);
    if (e != cudaSuccess) {
      g_cuda_error = e;
      (void)cudaGetLastError();
      delete p;
      g_status = e == cudaErrorMemoryAllocation ? FFT_ERR_ALLOC : FFT_ERR_CUDA;
      return nullptr;
    }
  }
  return p;
}

void fft_plan_destroy(fft_plan *plan) {
  if (!plan) return;
  if (plan->workspace) cudaFree(plan->workspace);
  if (plan->chirp) cudaFree(plan->chirp);
  if (plan->rtw) cudaFree(plan->rtw);
  if (plan->mtw) cudaFree(plan->mtw);
  if (plan->inner) fft_plan_destroy(plan->inner);
  for (int k = 0; k < 3; ++k)
    if (plan->axis_plan[k]) fft_plan_destroy(plan->axis_plan[k]);
  delete plan;
}

size_t fft_plan_workspace_bytes(const fft_plan *plan) {
  if (!plan) return 0;
  size_t b = plan->workspace_bytes + plan->aux_bytes + fft_plan_workspace_bytes(plan->inner);
  for (int k = 0; k < 3; ++k) b += fft_plan_workspace_bytes(plan->axis_plan[k]);
  return b;
}

}  // extern "C"
