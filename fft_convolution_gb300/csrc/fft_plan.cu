// fft_plan.cu -- host side of the library: plans, argument checks, the
// choice of kernels, and the exported C ABI declared in include/fft_gb300.h.
//
// The pages' own boundary is `solve(signal, spectrum, N)` on interleaved
// fp32 device buffers ("FFT on GPU", section FFT on GPU), which launches one
// kernel per butterfly stage with a device-wide synchronisation after each.
// Here a plan fixes the kernel sequence once; fft_exec only enqueues it on
// the caller's stream (1 kernel for on-chip lengths, 2 for 2D, 2-4 for long
// 1D transforms) and never synchronises.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>

#include "../../include/fft_gb300.h"
#include "internal.h"

using namespace fftgb;

// Device status word of the bounded in-kernel waits (0 = no error).
static __device__ int g_device_status;

namespace fftgb {
int *device_status_word() {
  static std::atomic<int *> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int *w = cache[dev].load(std::memory_order_acquire);
  if (!w) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) {
      w = static_cast<int *>(p);
      cache[dev].store(w, std::memory_order_release);
    }
  }
  return w;
}
}  // namespace fftgb

namespace {

thread_local int g_status = FFT_OK;
thread_local cudaError_t g_cuda_error = cudaSuccess;

enum Kind {
  KIND_ROWS = 0,
  KIND_MULTI = 1,
  KIND_ND = 2,
  KIND_DFT = 3,
  KIND_BLUESTEIN = 4,
  KIND_REAL_ROWS = 5,  // real, N = 2H with H a power of two on chip: one kernel
  KIND_REAL_EVEN = 6,  // real, other even N: complex plan of length N/2 + pre/post kernel
  KIND_REAL_ODD = 7,   // real, odd N: complex plan of length N + widen/narrow kernels
  KIND_MIXED = 8,      // N = 2^a 3^b 5^c 7^d (not a power of two) on chip
  KIND_ND_ANY = 9,     // 2D / 3D with a side that is not a power of two (or beyond KIND_ND's limits)
  KIND_FOUR_STEP = 10  // N = N1 N2 (2, 3, 5, 7 only) beyond one block: two mixed-radix plans
};

// Lengths that are not powers of two: the direct DFT up to this length,
// Bluestein beyond.
constexpr int64_t kDirectDftMax = 64;

constexpr int kMaxPasses = 8;

int ilog2_exact(int64_t n) {
  int l = 0;
  while (((int64_t)1 << l) < n) ++l;
  return l;
}

bool is_pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }

// Records a failed CUDA call and consumes the runtime's last-error state it
// left (a failed allocation would otherwise surface again at the next
// launch check of an unrelated call).
int cuda_fail(cudaError_t e) {
  g_cuda_error = e;
  (void)cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? FFT_ERR_ALLOC : FFT_ERR_CUDA;
}

bool misaligned(const void *p) { return ((uintptr_t)p & 15u) != 0; }

// Largest on-chip factor (log2) per HBM pass of a long 1D transform.  The
// default 9 keeps every pass tile at 64 KB with 16 (fp32) / 8 (fp64)
// contiguous columns; FFT_GB300_PASS_LOG overrides it (4 .. 14 fp32,
// 4 .. 13 fp64) for tuning.
int pass_log_limit(int dtype) {
  int lim = 9;
  const char *env = getenv("FFT_GB300_PASS_LOG");
  if (env && *env) {
    int v = atoi(env);
    if (v >= 4) lim = v;
  }
  const int hard = dtype == FFT_C2C_F32 ? kPassMaxLogF32 : kPassMaxLogF64;
  return lim > hard ? hard : lim;
}

// Bytes of data an L2-grouped schedule keeps in flight between two
// dependent kernels so that the second finds the first's output in L2.
// Measured on GB300, grouping 2D images (32 MiB) or fusing the first two
// passes of a 2^26 transform by 32 MiB groups is slower than whole-array
// passes (more, smaller launches with partial last waves), so grouping is
// off by default (0) and FFT_GB300_L2_BYTES turns it on for tuning.
size_t l2_group_bytes() {
  size_t v = 0;
  const char *env = getenv("FFT_GB300_L2_BYTES");
  if (env && *env) {
    long long x = atoll(env);
    if (x > 0) v = (size_t)x;
  }
  return v;
}

cudaError_t launch_rows(int dtype, int logn, int dir, const void *in, void *out, long long batch,
                        cudaStream_t st) {
  return dtype == FFT_C2C_F32 ? launch_rows_f32(logn, dir, in, out, batch, st)
                              : launch_rows_f64(logn, dir, in, out, batch, st);
}

cudaError_t launch_pass(int dtype, int dir, const PassArgs &a, const void *in, void *out,
                        cudaStream_t st) {
  return dtype == FFT_C2C_F32 ? launch_pass_f32(dir, a, in, out, st)
                              : launch_pass_f64(dir, a, in, out, st);
}

}  // namespace

struct fft_plan {
  int64_t n;      // 1D: the length; ND: the innermost (contiguous) side
  int64_t batch;
  int64_t elems;  // elements per transform (n, or the product of the sides)
  int rank;       // 1, 2 or 3
  int shape_log[3];  // log2 of the sides, outermost first (ND)
  int dims;
  int direction;
  int dtype;
  int kind;
  int logn;
  int npasses;
  int pass_log[kMaxPasses];
  void *workspace;
  size_t workspace_bytes;
  // Bluestein: convolution length 2^log_m; chirp (n values) and the filter
  // spectrum (2^log_m values) in one allocation.
  int log_m;
  void *chirp;
  void *filter;
  size_t aux_bytes;
  // Real sequences (FFT_REAL_*; dtype then holds the matching complex type).
  int real;
  fft_plan *inner;     // the complex plan of KIND_REAL_EVEN / KIND_REAL_ODD
  size_t ws_stride;    // workspace bytes per transform (batch ranges slice it)
  void *rtw;           // split twiddle table of W_N (KIND_REAL_EVEN), in aux
  int rtw_log_s;
  int64_t rtw_nhi;
  // Mixed radix: the stages and their forward twiddle table (in aux).
  MixedStages ms;
  void *mtw;
  // KIND_ND_ANY: the sides (outermost first), and per axis either a 1D plan
  // of any length (run on the contiguous axis, or between two transposes)
  // or an in-place power-of-two column pass (axis_pass).
  int64_t side[3];
  fft_plan *axis_plan[3];
  int axis_pass[3];
  // KIND_ND with every axis as on-chip rows stored transposed (nd_rows_t).
  int nd_rows_t;
};

namespace {

size_t complex_bytes(const fft_plan *p) { return p->dtype == FFT_C2C_F32 ? 8 : 16; }

// Bytes of one transform's input and output.
size_t in_tbytes(const fft_plan *p) {
  if (!p->real) return (size_t)p->elems * complex_bytes(p);
  return p->direction < 0 ? (size_t)p->n * (complex_bytes(p) / 2)
                          : (size_t)(p->n / 2 + 1) * complex_bytes(p);
}
size_t out_tbytes(const fft_plan *p) {
  if (!p->real) return (size_t)p->elems * complex_bytes(p);
  return p->direction < 0 ? (size_t)(p->n / 2 + 1) * complex_bytes(p)
                          : (size_t)p->n * (complex_bytes(p) / 2);
}

// Workspace bytes that belong to one transform (0: the plan's workspace is
// reused whole by every batch range on one stream, as Bluestein's is).
size_t ws_tbytes(const fft_plan *p) {
  if (p->kind == KIND_MULTI) return (size_t)p->n * complex_bytes(p);
  if (p->kind == KIND_REAL_EVEN || p->kind == KIND_REAL_ODD || p->kind == KIND_ND_ANY ||
      p->kind == KIND_FOUR_STEP || (p->kind == KIND_ND && p->nd_rows_t))
    return p->ws_stride;
  return 0;
}

cudaError_t launch_real_rows(int dtype, int logh, int dir, const void *in, void *out,
                             long long batch, cudaStream_t st) {
  return dtype == FFT_C2C_F32 ? launch_real_rows_f32(logh, dir, in, out, batch, st)
                              : launch_real_rows_f64(logh, dir, in, out, batch, st);
}

cudaError_t real_aux(int dtype, int op, const RealAuxArgs &a, cudaStream_t st) {
  return dtype == FFT_C2C_F32 ? real_aux_f32(op, a, st) : real_aux_f64(op, a, st);
}

}  // namespace

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

// The stages of a mixed-radix plan of length n: the odd factors first (3s,
// then 5s, then 7s: short blocks m while the stride N/R is odd), then the
// power of two as one 2, 4 or 8 and radix-16 stages.  False if n has a prime
// factor above 7 or needs more than 16 stages.
static bool mixed_stages(int64_t n, int elem, MixedStages *ms) {
  int radix[64], k = 0, a = 0;
  int64_t r = n;
  while (r % 2 == 0) {
    r /= 2;
    ++a;
  }
  const int odd[3] = {3, 5, 7};
  for (int f : odd)
    while (r % f == 0 && k < 64) {
      r /= f;
      radix[k++] = f;
    }
  if (r != 1) return false;
  if (a % 4) radix[k++] = 1 << (a % 4);
  for (int j = 0; j < a / 4; ++j) radix[k++] = 16;
  if (k > 16) return false;
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

static bool is_smooth_2357(int64_t n) {
  const int f[4] = {2, 3, 5, 7};
  for (int k = 0; k < 4; ++k)
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
// chip for longer lengths whose prime factors are 2, 3, 5, 7 (up to
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
  if (n > mixed_max && is_smooth_2357(n)) {
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
// shorter ones (64^3 x 256: 0.649 vs 0.540).  FFT_GB300_ND_ROWS_T=0 / 1
// forces the choice (sides 2^4 .. the transposed-store limit) for tuning.
static int nd_rows_t_wanted(int rank, const int *logs, int dtype) {
  const int lim = dtype == FFT_C2C_F32 ? rows_t_max_log_f32() : rows_t_max_log_f64();
  int ok = 1, preferred = 1;
  for (int k = 0; k < rank; ++k) {
    if (logs[k] < 4 || logs[k] > lim) ok = 0;
    if (logs[k] < 7 || logs[k] > 8) preferred = 0;
  }
  const char *env = getenv("FFT_GB300_ND_ROWS_T");
  if (env && *env) return ok && atoi(env) != 0;
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
  // most pass_log_limit bits, larger factors first.
  const int lim = pass_log_limit(dtype);
  int P = (logn + lim - 1) / lim;
  if (P < 2) P = 2;
  if (P > kMaxPasses) {
    delete p;
    g_status = FFT_ERR_UNSUPPORTED;
    return nullptr;
  }
  p->kind = KIND_MULTI;
  p->npasses = P;
  for (int k = 0; k < P; ++k) p->pass_log[k] = logn / P + (k < logn % P ? 1 : 0);
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

namespace {

// Enqueues (or, with dry = true, only counts) the kernels of one fft_exec.
struct Schedule {
  const fft_plan *p;
  cudaStream_t st;
  bool dry;
  long long batch;  // transforms this run covers: b0 .. b0 + batch - 1 of the plan's
  long long b0;
  int count = 0;
  char *ws = nullptr;  // the workspace slice of that range

  Schedule(const fft_plan *p_, cudaStream_t st_, bool dry_, long long batch_, long long b0_)
      : p(p_), st(st_), dry(dry_), batch(batch_), b0(b0_) {
    if (p->workspace) ws = static_cast<char *>(p->workspace) + (size_t)b0 * ws_tbytes(p);
  }

  size_t elem() const { return p->dtype == FFT_C2C_F32 ? 8 : 16; }

  cudaError_t rows(const void *in, void *out, long long nrows) {
    ++count;
    return dry ? cudaSuccess : launch_rows(p->dtype, p->logn, p->direction, in, out, nrows, st);
  }
  cudaError_t pass(const PassArgs &a, const void *in, void *out) {
    ++count;
    return dry ? cudaSuccess : launch_pass(p->dtype, p->direction, a, in, out, st);
  }
  int tile_cols(int log_l) const {
    return p->dtype == FFT_C2C_F32 ? pass_tile_cols_f32(log_l) : pass_tile_cols_f64(log_l);
  }

  // 2D / 3D: rows (the contiguous side) on chip, then every other axis as
  // an in-place column pass (stride = the product of the inner sides), from
  // the inner axes outward.  With an L2 budget set, one L2-sized group of
  // transforms at a time so the column passes read the rows' output from L2.
  // KIND_ND with transposed-store rows: pass k transforms the contiguous
  // axis of [R][L] and writes [L][R]; after `rank` passes the order is the
  // original one.  Buffers: 2 passes in -> ws -> out; 3 passes in -> out ->
  // ws -> out (in place: in -> ws -> in -> ws, then a copy back).
  cudaError_t run_nd_rows_t(const char *in, char *out) {
    const int r = p->rank;
    int total_log = 0;
    for (int k = 0; k < r; ++k) total_log += p->shape_log[k];
    const char *src = in;
    cudaError_t e = cudaSuccess;
    for (int k = 0; k < r; ++k) {
      // Pass k: contiguous axis = original axis r-1-k.
      const int l = p->shape_log[r - 1 - k];
      char *dst;
      if (r == 2) {
        dst = k == 0 ? ws : out;
      } else if (in != out) {
        dst = k == 1 ? ws : out;
      } else {
        dst = k == 1 ? out : ws;
      }
      ++count;
      if (!dry) {
        const long long rows = batch << (total_log - l);
        e = p->dtype == FFT_C2C_F32
                ? launch_rows_t_f32(l, p->direction, src, dst, rows, total_log - l, st)
                : launch_rows_t_f64(l, p->direction, src, dst, rows, total_log - l, st);
        if (e != cudaSuccess) return e;
      }
      src = dst;
    }
    if (!dry && src != out)
      e = cudaMemcpyAsync(out, src, (size_t)batch * p->elems * elem(), cudaMemcpyDeviceToDevice, st);
    return e;
  }

  cudaError_t run_nd(const char *in, char *out) {
    if (p->nd_rows_t) return run_nd_rows_t(in, out);
    const size_t tbytes = (size_t)p->elems * elem();
    const size_t budget = l2_group_bytes();
    long long g = budget ? (long long)(budget / tbytes) : batch;
    if (g < 1) g = 1;
    for (long long b0 = 0; b0 < batch; b0 += g) {
      const long long nb = batch - b0 < g ? batch - b0 : g;
      const size_t off = (size_t)b0 * tbytes;
      cudaError_t e = rows(in + off, out + off, nb * (p->elems >> p->logn));
      if (e != cudaSuccess) return e;
      int inner = p->logn;  // log2 of the stride of the next axis
      for (int k = p->rank - 2; k >= 0; --k) {
        const int l = p->shape_log[k];
        if (l > 0) {
          const int log_block = l + inner;  // one column block: L * stride elements
          PassArgs a{log_block, l, inner, 0, nb * (p->elems >> log_block), {}};
          e = pass(a, out + off, out + off);
          if (e != cudaSuccess) return e;
        }
        inner += l;
      }
    }
    return cudaSuccess;
  }

  // KIND_ND_ANY (see plan_nd_any), over this range of the batch.
  cudaError_t run_nd_any(const char *in, char *out) {
    const int64_t total = p->elems;
    const size_t elem = this->elem();
    const int r = p->rank;
    cudaError_t e = cudaSuccess;
    // Contiguous axis: in -> out.
    if (p->axis_plan[r - 1]) {
      const long long rows = total / p->side[r - 1];
      Schedule s1(p->axis_plan[r - 1], st, dry, batch * rows, b0 * rows);
      e = s1.run(in, out);
      count += s1.count;
      if (e != cudaSuccess) return e;
    } else if (in != out && !dry) {  // contiguous side of length 1: the data moves as is
      e = cudaMemcpyAsync(out, in, (size_t)batch * total * elem, cudaMemcpyDeviceToDevice, st);
      if (e != cudaSuccess) return e;
    }
    int64_t stride = p->side[r - 1];
    for (int k = r - 2; k >= 0; --k) {
      const int64_t L = p->side[k];
      const long long outer = batch * (total / (L * stride));
      if (p->axis_pass[k]) {
        const int l = ilog2_exact(L), inner = ilog2_exact(stride);
        PassArgs a{l + inner, l, inner, 0, outer, {}};
        e = pass(a, out, out);
      } else if (p->axis_plan[k]) {
        // [outer][L][stride] -> ws [outer][stride][L], transform, and back.
        count += 2;
        if (!dry) e = transpose_complex(p->dtype == FFT_C2C_F64, out, ws, outer, L, stride, st);
        if (e != cudaSuccess) return e;
        const long long rows = total / L;
        Schedule sk(p->axis_plan[k], st, dry, batch * rows, b0 * rows);
        e = sk.run(ws, ws);
        count += sk.count;
        if (e != cudaSuccess) return e;
        if (!dry) e = transpose_complex(p->dtype == FFT_C2C_F64, ws, out, outer, stride, L, st);
      }
      if (e != cudaSuccess) return e;
      stride *= L;
    }
    return cudaSuccess;
  }

  // KIND_FOUR_STEP (see plan_four_step) over this range of the batch.  Out
  // of place: in -> out (transpose), out (length n1), out -> ws (twiddled
  // transpose), ws (length n2), ws -> out (transpose).  In place the first
  // transpose goes to ws and the last result comes back by a copy.
  cudaError_t run_four_step(const char *in, char *out) {
    const int64_t n1 = p->side[0], n2 = p->side[1];
    const int f64 = p->dtype == FFT_C2C_F64;
    const size_t elem = this->elem();
    const char *lo = static_cast<const char *>(p->rtw);
    const char *hi = lo + ((size_t)1 << p->rtw_log_s) * elem;
    char *a = in != out ? out : ws;  // holds [n2][k1] after the first two steps
    char *b = in != out ? ws : out;  // holds [k1][k2] after the next two
    cudaError_t e = cudaSuccess;
    count += 3;
    if (!dry) e = transpose_complex(f64, in, a, batch, n1, n2, st);
    if (e != cudaSuccess) return e;
    Schedule s1(p->axis_plan[0], st, dry, batch * n2, b0 * n2);
    if ((e = s1.run(a, a)) != cudaSuccess) return e;
    count += s1.count;
    if (!dry)
      e = transpose_twiddle_complex(f64, a, b, batch, n2, n1, p->n, lo, hi, p->rtw_log_s,
                                    p->direction > 0, st);
    if (e != cudaSuccess) return e;
    Schedule s2(p->axis_plan[1], st, dry, batch * n1, b0 * n1);
    if ((e = s2.run(b, b)) != cudaSuccess) return e;
    count += s2.count;
    if (dry) return cudaSuccess;
    if (in != out) return transpose_complex(f64, b, out, batch, n1, n2, st);
    if ((e = transpose_complex(f64, b, ws, batch, n1, n2, st)) != cudaSuccess) return e;
    return cudaMemcpyAsync(out, ws, (size_t)batch * p->n * elem, cudaMemcpyDeviceToDevice, st);
  }

  // Passes k_begin.. of `batch` transforms.  Pass k reads the previous
  // pass's output; intermediates alternate between the workspace and `out`
  // and the last pass always writes `out` (it reads and writes the same
  // positions, so in place is safe).
  cudaError_t run_passes(const char *in, char *out, char *ws, long long batch, int k_begin) {
    int log_m = 0;
    for (int k = 0; k < k_begin; ++k) log_m += p->pass_log[k];
    const char *src = k_begin == 0 ? in : (k_begin % 2 == 1 ? ws : out);
    for (int k = k_begin; k < p->npasses; ++k) {
      char *dst = (k == p->npasses - 1) ? out : (k % 2 == 0 ? ws : out);
      PassArgs a{p->logn, p->pass_log[k], log_m, 1, batch, {}};
      cudaError_t e = pass(a, src, dst);
      if (e != cudaSuccess) return e;
      src = dst;
      log_m += p->pass_log[k];
    }
    return cudaSuccess;
  }

  // Passes 0 and 1 of one transform fused through L2.  Pass-1 butterfly
  // q*L0 + p (q < Q = N/(L0 L1)) reads exactly the outputs of the pass-0
  // butterflies q + u*Q (u < L1), so for a group of G consecutive q both
  // passes close over G*L0*L1 elements: run pass 0 for the group (its
  // output stays in L2), then pass 1 for the group, group after group.
  // Returns false (nothing launched) when the sizes do not allow it.
  bool fused_01(const char *in, char *out, char *ws, cudaError_t *err) {
    const int l0 = p->pass_log[0], l1 = p->pass_log[1];
    const long long L0 = 1LL << l0, L1 = 1LL << l1;
    const long long Q = 1LL << (p->logn - l0 - l1);
    const long long C0 = tile_cols(l0), C1 = tile_cols(l1);
    long long G = (long long)(l2_group_bytes() / ((size_t)L0 * L1 * elem()));
    if (G < C0) G = C0;
    while (G & (G - 1)) G &= G - 1;  // power of two
    if (C0 <= 0 || C1 <= 0 || Q < C0 || G > Q || Q % G || (G * L0) % C1) return false;
    for (long long q0 = 0; q0 < Q; q0 += G) {
      PassArgs a0{p->logn, l0, 0, 1, 1, {q0 / C0, G / C0, Q / C0, L1}};
      *err = pass(a0, in, ws);
      if (*err != cudaSuccess) return true;
      PassArgs a1{p->logn, l1, l0, 1, 1, {q0 * L0 / C1, G * L0 / C1, 0, 1}};
      *err = pass(a1, ws, out);
      if (*err != cudaSuccess) return true;
    }
    *err = cudaSuccess;
    return true;
  }

  cudaError_t run_multi(const char *in, char *out) {
    const size_t tbytes = (size_t)p->n * elem();
    const size_t budget = l2_group_bytes();
    if (budget == 0) return run_passes(in, out, ws, batch, 0);
    if (tbytes <= budget) {
      // Whole transforms fit in L2: all passes of one group, then the next.
      long long g = (long long)(budget / tbytes);
      if (g < 1) g = 1;
      for (long long b0 = 0; b0 < batch; b0 += g) {
        const long long nb = batch - b0 < g ? batch - b0 : g;
        const size_t off = (size_t)b0 * tbytes;
        cudaError_t e = run_passes(in + off, out + off, ws + off, nb, 0);
        if (e != cudaSuccess) return e;
      }
      return cudaSuccess;
    }
    // Larger than L2: fuse the first two passes through L2 when the result
    // may not overwrite the input early (out of place) and there is a pass
    // left to run after them.
    if (in != out && p->npasses >= 3) {
      bool fused = true;
      for (long long b = 0; b < batch && fused; ++b) {
        const size_t off = (size_t)b * tbytes;
        cudaError_t e = cudaSuccess;
        fused = fused_01(in + off, out + off, ws + off, &e);
        if (e != cudaSuccess) return e;
      }
      if (fused) return run_passes(in, out, ws, batch, 2);
    }
    return run_passes(in, out, ws, batch, 0);
  }

  cudaError_t run(const void *in, void *out) {
    const char *i = static_cast<const char *>(in);
    char *o = static_cast<char *>(out);
    switch (p->kind) {
      case KIND_ROWS:
        return rows(in, out, batch);
      case KIND_ND:
        return run_nd(i, o);
      case KIND_ND_ANY:
        return run_nd_any(i, o);
      case KIND_FOUR_STEP:
        return run_four_step(i, o);
      case KIND_DFT: {
        ++count;
        if (dry) return cudaSuccess;
        const double scale = p->direction > 0 ? 1.0 / (double)p->n : 1.0;
        return p->dtype == FFT_C2C_F32
                   ? dft_small_f32(in, out, (int)p->n, batch, p->direction, scale, st)
                   : dft_small_f64(in, out, (int)p->n, batch, p->direction, scale, st);
      }
      case KIND_BLUESTEIN: {
        const int on_chip = p->dtype == FFT_C2C_F32 ? RowsMaxLog<float>::value
                                                    : RowsMaxLog<double>::value;
        // Fused: one kernel.  Multi-pass: the forward and inverse passes of
        // the convolution (its filter spectrum was computed at planning).
        count += p->log_m <= on_chip ? 1 : 2 * convolve_passes(p->dtype, p->log_m);
        if (dry) return cudaSuccess;
        const double scale = p->direction > 0 ? 1.0 / (double)p->n : 1.0;
        // The work arrays are reused chunk after chunk (one stream), so the
        // plan's own base is used for any batch range.
        return p->dtype == FFT_C2C_F32
                   ? bluestein_exec_f32(in, out, p->n, batch, p->log_m, scale, p->chirp, p->filter,
                                        p->workspace, st)
                   : bluestein_exec_f64(in, out, p->n, batch, p->log_m, scale, p->chirp, p->filter,
                                        p->workspace, st);
      }
      case KIND_MULTI:
        return run_multi(i, o);
      case KIND_MIXED:
        ++count;
        if (dry) return cudaSuccess;
        return p->dtype == FFT_C2C_F32
                   ? mixed_exec_f32(in, out, batch, p->ms, p->mtw, p->direction, st)
                   : mixed_exec_f64(in, out, batch, p->ms, p->mtw, p->direction, st);
      case KIND_REAL_ROWS:
        ++count;
        return dry ? cudaSuccess : launch_real_rows(p->dtype, p->logn, p->direction, in, out, batch, st);
      case KIND_REAL_EVEN:
      case KIND_REAL_ODD:
        return run_real(in, out);
      default:
        return cudaErrorInvalidValue;
    }
  }

  // Real sequences around the inner complex plan (same batch range).  Even
  // N: forward = complex transform of the samples read as N/2 complex values
  // into the workspace, then the post kernel; inverse = pre kernel into the
  // workspace, then the complex inverse into `out`.  Odd N: samples widened
  // into the workspace, transformed there in place, bins 0 .. N/2 copied out
  // (forward); spectrum extended into the workspace, inverse in place, real
  // parts copied out (inverse).
  cudaError_t run_real(const void *in, void *out) {
    Schedule inner(p->inner, st, dry, batch, b0);
    const bool even = p->kind == KIND_REAL_EVEN;
    const size_t elem = complex_bytes(p);
    const char *lo = static_cast<const char *>(p->rtw);
    const char *hi = lo ? lo + ((size_t)1 << p->rtw_log_s) * elem : nullptr;
    const long long len = even ? p->n / 2 : p->n;
    auto aux = [&](int op, const void *a_in, void *a_out) -> cudaError_t {
      ++count;
      if (dry) return cudaSuccess;
      RealAuxArgs a{a_in, a_out, len, batch, lo, hi, p->rtw_log_s, p->rtw_nhi};
      return real_aux(p->dtype, op, a, st);
    };
    cudaError_t e;
    if (p->direction < 0) {
      if (even) {
        e = inner.run(in, ws);
      } else {
        if ((e = aux(REAL_WIDEN, in, ws)) != cudaSuccess) return e;
        e = inner.run(ws, ws);
      }
      count += inner.count;
      if (e != cudaSuccess) return e;
      return aux(even ? REAL_POST : REAL_NARROW, ws, out);
    }
    if ((e = aux(even ? REAL_PRE : REAL_EXTEND, in, ws)) != cudaSuccess) return e;
    e = even ? inner.run(ws, out) : inner.run(ws, ws);
    count += inner.count;
    if (e != cudaSuccess || even) return e;
    return aux(REAL_PART, ws, out);
  }
};

}  // namespace

extern "C" {

int fft_plan_num_kernels(const fft_plan *plan) {
  if (!plan) return 0;
  // Count an out-of-place execution (distinct dummy addresses).
  Schedule s(plan, nullptr, true, plan->batch, 0);
  s.run(reinterpret_cast<const void *>(16), reinterpret_cast<void *>(32));
  return s.count;
}

int fft_exec(const fft_plan *p, const void *in, void *out, void *stream) {
  if (!p || !in || !out) return FFT_ERR_INVALID_ARG;
  if (p->real && in == out) return FFT_ERR_INVALID_ARG;  // sizes differ: out of place only
  if (misaligned(in) || misaligned(out)) return FFT_ERR_MISALIGNED;
  Schedule s(p, static_cast<cudaStream_t>(stream), false, p->batch, 0);
  cudaError_t e = s.run(in, out);
  if (e != cudaSuccess) return cuda_fail(e);
  return FFT_OK;
}

int fft_exec_host(const fft_plan *p, const void *host_in, void *host_out, void *dev_in,
                  void *dev_out, void *stream) {
  if (!p || !dev_in || !dev_out) return FFT_ERR_INVALID_ARG;
  if (misaligned(dev_in) || misaligned(dev_out)) return FFT_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (host_in) {
    e = cudaMemcpyAsync(dev_in, host_in, (size_t)p->batch * in_tbytes(p), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  int rc = fft_exec(p, dev_in, dev_out, stream);
  if (rc != FFT_OK) return rc;
  if (host_out) {
    e = cudaMemcpyAsync(host_out, dev_out, (size_t)p->batch * out_tbytes(p), cudaMemcpyDeviceToHost,
                        st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return FFT_OK;
}

}  // extern "C"

namespace {

// Streams and events of the host-staged pipeline, created once per device.
struct HostPipe {
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t fork = nullptr, join_comp = nullptr, join_out = nullptr;
  cudaEvent_t *loaded = nullptr, *done = nullptr;  // per chunk
  int nev = 0;
};
std::mutex g_pipe_mutex;
HostPipe g_pipes[64];

cudaError_t pipe_for_device(int chunks, HostPipe **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  HostPipe &hp = g_pipes[dev];
  if (!hp.in) {
    const unsigned f = cudaStreamNonBlocking;
    if ((e = cudaStreamCreateWithFlags(&hp.in, f)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&hp.comp, f)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&hp.out, f)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.fork, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.join_comp, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.join_out, cudaEventDisableTiming)) != cudaSuccess)
      return e;
  }
  if (hp.nev < chunks) {
    cudaEvent_t *l = new (std::nothrow) cudaEvent_t[chunks];
    cudaEvent_t *d = new (std::nothrow) cudaEvent_t[chunks];
    if (!l || !d) {
      delete[] l;
      delete[] d;
      return cudaErrorMemoryAllocation;
    }
    for (int k = 0; k < hp.nev; ++k) {
      l[k] = hp.loaded[k];
      d[k] = hp.done[k];
    }
    for (int k = hp.nev; k < chunks; ++k) {
      if ((e = cudaEventCreateWithFlags(&l[k], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&d[k], cudaEventDisableTiming)) != cudaSuccess) {
        delete[] l;
        delete[] d;
        return e;
      }
    }
    delete[] hp.loaded;
    delete[] hp.done;
    hp.loaded = l;
    hp.done = d;
    hp.nev = chunks;
  }
  *out = &hp;
  return cudaSuccess;
}

// Streams `batch` items through the device in chunks of `chunk`: for each
// chunk, up() on the upload stream, compute() on the compute stream once the
// upload is done, down() on the download stream once the compute is done;
// forked from and joined back to `st`.  Each callback gets (first item,
// count, stream) and returns a cudaError_t.  Calls on one device enqueue
// under one lock (the pipeline's streams and events are shared).
template <class Up, class Comp, class Down>
int host_pipeline(long long batch, long long chunk, cudaStream_t st, Up up, Comp compute,
                  Down down) {
  if (chunk > batch) chunk = batch;
  const long long nchunks = (batch + chunk - 1) / chunk;
  if (nchunks > 4096) return FFT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  HostPipe *hp = nullptr;
  cudaError_t e = pipe_for_device((int)nchunks, &hp);
  if (e != cudaSuccess) return cuda_fail(e);
  // Fork: the three pipeline streams start after the work already on `st`.
  if ((e = cudaEventRecord(hp->fork, st)) != cudaSuccess) return cuda_fail(e);
  cudaStreamWaitEvent(hp->in, hp->fork, 0);
  cudaStreamWaitEvent(hp->comp, hp->fork, 0);
  cudaStreamWaitEvent(hp->out, hp->fork, 0);
  for (long long k = 0; k < nchunks; ++k) {
    const long long b0 = k * chunk;
    const long long cnt = batch - b0 < chunk ? batch - b0 : chunk;
    if ((e = up(b0, cnt, hp->in)) != cudaSuccess) return cuda_fail(e);
    cudaEventRecord(hp->loaded[k], hp->in);
    cudaStreamWaitEvent(hp->comp, hp->loaded[k], 0);
    if ((e = compute(b0, cnt, hp->comp)) != cudaSuccess) return cuda_fail(e);
    cudaEventRecord(hp->done[k], hp->comp);
    cudaStreamWaitEvent(hp->out, hp->done[k], 0);
    if ((e = down(b0, cnt, hp->out)) != cudaSuccess) return cuda_fail(e);
  }
  // Join: `st` continues after the last download.
  cudaEventRecord(hp->join_comp, hp->comp);
  cudaEventRecord(hp->join_out, hp->out);
  cudaStreamWaitEvent(st, hp->join_comp, 0);
  e = cudaStreamWaitEvent(st, hp->join_out, 0);
  if (e != cudaSuccess) return cuda_fail(e);
  return FFT_OK;
}

}  // namespace

extern "C" {

int fft_exec_host_chain(const fft_plan *const *plans, int nplans, const void *host_in,
                        void *host_out, void *dev_a, void *dev_b, int64_t chunk, void *stream) {
  if (!plans || nplans <= 0 || !host_in || !host_out || !dev_a || !dev_b || chunk <= 0)
    return FFT_ERR_INVALID_ARG;
  const fft_plan *p0 = plans[0];
  for (int k = 0; k < nplans; ++k) {
    const fft_plan *q = plans[k];
    // One batch; each plan takes what the previous one produces.
    if (!q || q->batch != p0->batch || (k > 0 && in_tbytes(q) != out_tbytes(plans[k - 1])))
      return FFT_ERR_INVALID_ARG;
  }
  if (misaligned(dev_a) || misaligned(dev_b)) return FFT_ERR_MISALIGNED;
  const long long batch = p0->batch;
  if (chunk > batch) chunk = batch;
  // Every chunk's slices must start 16-byte aligned, like whole buffers.
  for (int k = 0; k < nplans; ++k)
    if (((size_t)chunk * in_tbytes(plans[k])) % 16 || ((size_t)chunk * out_tbytes(plans[k])) % 16 ||
        ((size_t)chunk * ws_tbytes(plans[k])) % 16)
      return FFT_ERR_MISALIGNED;
  for (int k = 0; k < nplans; ++k)
    if (plans[k]->real && dev_a == dev_b) return FFT_ERR_INVALID_ARG;  // real: out of place only
  const size_t in_bytes0 = in_tbytes(p0), out_bytes_last = out_tbytes(plans[nplans - 1]);
  char *bufs[2] = {static_cast<char *>(dev_a), static_cast<char *>(dev_b)};
  return host_pipeline(
      batch, chunk, static_cast<cudaStream_t>(stream),
      [&](long long b0, long long cnt, cudaStream_t s) {
        return cudaMemcpyAsync(bufs[0] + (size_t)b0 * in_bytes0,
                               static_cast<const char *>(host_in) + (size_t)b0 * in_bytes0,
                               (size_t)cnt * in_bytes0, cudaMemcpyHostToDevice, s);
      },
      [&](long long b0, long long cnt, cudaStream_t s) {
        for (int j = 0; j < nplans; ++j) {
          const fft_plan *q = plans[j];
          Schedule sc(q, s, false, cnt, b0);
          cudaError_t e = sc.run(bufs[j % 2] + (size_t)b0 * in_tbytes(q),
                                 bufs[(j + 1) % 2] + (size_t)b0 * out_tbytes(q));
          if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
      },
      [&](long long b0, long long cnt, cudaStream_t s) {
        return cudaMemcpyAsync(static_cast<char *>(host_out) + (size_t)b0 * out_bytes_last,
                               bufs[nplans % 2] + (size_t)b0 * out_bytes_last,
                               (size_t)cnt * out_bytes_last, cudaMemcpyDeviceToHost, s);
      });
}

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

const char *fft_status_string(int status) {
  switch (status) {
    case FFT_OK: return "ok";
    case FFT_ERR_INVALID_ARG: return "invalid argument";
    case FFT_ERR_NOT_POW2: return "length is not a power of two";
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
