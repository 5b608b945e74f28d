// plan.h -- host-side internals shared by the library's C ABI translation
// units: the plan record, its kinds, the per-thread status, sizes of one
// transform's input / output / workspace, and the three-stream host
// pipeline.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <mutex>

#include "../../include/fft_gb300.h"
#include "internal.h"

namespace fftgb {

// Status of the last call on this thread (fft_last_status) and the CUDA
// error behind an FFT_ERR_CUDA / FFT_ERR_ALLOC (fft_last_cuda_error).
extern thread_local int g_status;
extern thread_local cudaError_t g_cuda_error;

enum Kind {
  KIND_ROWS = 0,
  KIND_MULTI = 1,
  KIND_ND = 2,
  KIND_DFT = 3,
  KIND_BLUESTEIN = 4,
  KIND_REAL_ROWS = 5,  // real, N = 2H with H a power of two on chip: one kernel
  KIND_REAL_EVEN = 6,  // real, other even N: complex plan of length N/2 + pre/post kernel
  KIND_REAL_ODD = 7,   // real, odd N: complex plan of length N + widen/narrow kernels
  KIND_MIXED = 8,      // N = 2^a 3^b 5^c 7^d 11^e 13^f (not a power of two) on chip
  KIND_ND_ANY = 9,     // 2D / 3D with a side that is not a power of two (or beyond KIND_ND's limits)
  KIND_FOUR_STEP = 10  // N = N1 N2 (factors 2 .. 13 only) beyond one block: two mixed-radix plans
};

// Lengths that are not powers of two: the direct DFT up to this length,
// Bluestein beyond.
constexpr int64_t kDirectDftMax = 64;

constexpr int kMaxPasses = 8;

inline int ilog2_exact(int64_t n) {
  int l = 0;
  while (((int64_t)1 << l) < n) ++l;
  return l;
}

inline bool is_pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }

// Records a failed CUDA call and consumes the runtime's last-error state it
// left (a failed allocation would otherwise surface again at the next
// launch check of an unrelated call).
int cuda_fail(cudaError_t e);

inline bool misaligned(const void *p) { return ((uintptr_t)p & 15u) != 0; }

// Largest on-chip factor (log2) per HBM pass of a long 1D plan (fft_plan.cu).
int pass_log_limit(int dtype);

inline cudaError_t launch_rows(int dtype, int logn, int dir, const void *in, void *out,
                               long long batch, cudaStream_t st) {
  return dtype == FFT_C2C_F32 ? launch_rows_f32(logn, dir, in, out, batch, st)
                              : launch_rows_f64(logn, dir, in, out, batch, st);
}

inline cudaError_t launch_pass(int dtype, int dir, const PassArgs &a, const void *in, void *out,
                               cudaStream_t st) {
  return dtype == FFT_C2C_F32 ? launch_pass_f32(dir, a, in, out, st)
                              : launch_pass_f64(dir, a, in, out, st);
}

}  // namespace fftgb

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
  int pass_log[fftgb::kMaxPasses];
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
  void *rtw;           // split twiddle table of W_N (KIND_REAL_EVEN, KIND_FOUR_STEP), in aux
  int rtw_log_s;
  int64_t rtw_nhi;
  // Mixed radix: the stages and their forward twiddle table (in aux).
  fftgb::MixedStages ms;
  void *mtw;
  // KIND_ND_ANY: the sides (outermost first), and per axis either a 1D plan
  // of any length (run on the contiguous axis, or between two transposes)
  // or an in-place power-of-two column pass (axis_pass).  KIND_FOUR_STEP:
  // side[0] = N1, side[1] = N2 and their plans in axis_plan[0..1].
  int64_t side[3];
  fft_plan *axis_plan[3];
  int axis_pass[3];
  // KIND_ND with every axis as on-chip rows stored transposed (nd_rows_t).
  int nd_rows_t;
  // KIND_ND, out of place: log2 of the radix of the column transform's first
  // stage folded into the row pass (0: rows, then a full column pass).
  int col_radix_log;
};

namespace fftgb {

inline size_t complex_bytes(const fft_plan *p) { return p->dtype == FFT_C2C_F32 ? 8 : 16; }

// Bytes of one transform's input and output.
inline size_t in_tbytes(const fft_plan *p) {
  if (!p->real) return (size_t)p->elems * complex_bytes(p);
  return p->direction < 0 ? (size_t)p->n * (complex_bytes(p) / 2)
                          : (size_t)(p->n / 2 + 1) * complex_bytes(p);
}
inline size_t out_tbytes(const fft_plan *p) {
  if (!p->real) return (size_t)p->elems * complex_bytes(p);
  return p->direction < 0 ? (size_t)(p->n / 2 + 1) * complex_bytes(p)
                          : (size_t)p->n * (complex_bytes(p) / 2);
}

// Workspace bytes that belong to one transform (0: the plan's workspace is
// reused whole by every batch range on one stream, as Bluestein's is).
inline size_t ws_tbytes(const fft_plan *p) {
  if (p->kind == KIND_MULTI) return (size_t)p->n * complex_bytes(p);
  if (p->kind == KIND_REAL_EVEN || p->kind == KIND_REAL_ODD || p->kind == KIND_ND_ANY ||
      p->kind == KIND_FOUR_STEP || (p->kind == KIND_ND && p->nd_rows_t))
    return p->ws_stride;
  return 0;
}

inline cudaError_t launch_real_rows(int dtype, int logh, int dir, const void *in, void *out,
                             long long batch, cudaStream_t st) {
  return dtype == FFT_C2C_F32 ? launch_real_rows_f32(logh, dir, in, out, batch, st)
                              : launch_real_rows_f64(logh, dir, in, out, batch, st);
}

inline cudaError_t real_aux(int dtype, int op, const RealAuxArgs &a, cudaStream_t st) {
  return dtype == FFT_C2C_F32 ? real_aux_f32(op, a, st) : real_aux_f64(op, a, st);
}


// Streams and events of the host-staged pipeline, created once per device.
struct HostPipe {
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t fork = nullptr, join_comp = nullptr, join_out = nullptr;
  cudaEvent_t *loaded = nullptr, *done = nullptr;  // per chunk
  int nev = 0;
};
extern std::mutex g_pipe_mutex;
cudaError_t pipe_for_device(int chunks, HostPipe **out);

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

}  // namespace fftgb
