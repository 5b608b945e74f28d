// fft_exec.cu -- execution: the kernel schedule of every plan kind
// (fft_exec, fft_plan_num_kernels), host staging (fft_exec_host) and the
// chunked three-stream pipeline over host buffers (fft_exec_host_chain).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>

#include "plan.h"

using namespace fftgb;

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
    // Out of place with long columns: the row pass also takes the first
    // radix-R stage of the column transform (fft_rows_col.cuh), and the
    // column pass then has on-chip length H / R over columns R W apart.
    const int logr = in != out ? p->col_radix_log : 0;
    cudaError_t e;
    if (logr > 0) {
      const int logh = p->shape_log[p->rank - 2];
      ++count;
      e = dry ? cudaSuccess
              : (p->dtype == FFT_C2C_F32 ? launch_rows_col_f32 : launch_rows_col_f64)(
                    p->logn, logr, p->direction, in, out, logh,
                    batch * (p->elems >> (p->logn + logh)), st);
    } else {
      e = rows(in, out, batch * (p->elems >> p->logn));
    }
    if (e != cudaSuccess) return e;
    int inner = p->logn;  // log2 of the stride of the next axis
    int after_pass = 0;   // the previous kernel was a pass (not the row kernel)
    for (int k = p->rank - 2; k >= 0; --k) {
      int l = p->shape_log[k];
      int stride_log = inner;
      if (k == p->rank - 2 && logr > 0) {  // the rest of the folded column transform
        l -= logr;
        stride_log += logr;
      }
      if (l > 0) {
        const int log_block = l + stride_log;  // one column block: L * stride elements
        // The first column pass follows the row kernel; a later one (3D)
        // follows a pass and may overlap its tail.
        PassArgs a{log_block, l, stride_log, 0, batch * (p->elems >> log_block), after_pass};
        e = pass(a, out, out);
        if (e != cudaSuccess) return e;
        after_pass = 1;
      }
      inner += p->shape_log[k];
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
        PassArgs a{l + inner, l, inner, 0, outer};
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
      PassArgs a{p->logn, p->pass_log[k], log_m, 1, batch, k > 0 ? 1 : 0};
      cudaError_t e = pass(a, src, dst);
      if (e != cudaSuccess) return e;
      src = dst;
      log_m += p->pass_log[k];
    }
    return cudaSuccess;
  }

  cudaError_t run_multi(const char *in, char *out) { return run_passes(in, out, ws, batch, 0); }

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

namespace fftgb {

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

}  // namespace fftgb

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

}  // extern "C"
