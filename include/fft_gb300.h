/*
 * fft_gb300.h -- C ABI of the GB300 (sm_103a) FFT library.
 *
 * Operations (all on one GPU, asynchronous on the caller's CUDA stream):
 *   - batched 1D complex-to-complex transforms of any length, forward
 *     (unscaled) and inverse (scaled by 1/N), fp32 or fp64: powers of two on
 *     chip or in 2-4 HBM passes; other lengths by the direct DFT (N <= 64),
 *     mixed radix (prime factors 2, 3, 5, 7, 11, 13; four-step beyond one
 *     block) or
 *     Bluestein;
 *   - transforms of real sequences (half spectrum out / in, any length);
 *   - separable 2D and 3D transforms of any sides (rows, then columns, ...);
 *   - linear convolution of complex or real signals;
 *   - integer polynomial multiplication through fp64 transforms;
 *   - host-buffer forms of these, streamed through the device in chunks.
 *
 * Definitions followed:
 *   forward   X_k = sum_{n<N} x_n e^{-i 2 pi k n / N}
 *             ("FFT on GPU", elwhyjay.github.io/post/fft, section
 *             Discrete Fourier Transform)
 *   inverse   x_n = (1/N) sum_{k<N} X_k e^{+i 2 pi k n / N}
 *             (same page, polynomial-multiplication section: omega replaced
 *             by omega^{-1} and the factor 1/N)
 *   2D / 3D   1D transforms along every row, then along every column, ...
 *             ("Stockham FFT Butterfly Algorithm in Parallel GLSL",
 *             section Multi-Dimensional Transforms and Separability)
 *   polymul   c_k = sum_i a_i b_{k-i}, computed as transform, pointwise
 *             product of the point values, inverse transform ("FFT on GPU",
 *             polynomial-multiplication section, whole pipeline)
 *   convolve  y_k = sum_i x_i h_{k-i}, the same pipeline for signals
 *
 * Data layout: complex arrays are interleaved (re, im) pairs of float
 * (FFT_C2C_F32) or double (FFT_C2C_F64) -- the layout of the pages' CUDA
 * code, and of torch.complex64 / torch.complex128.  A batch is contiguous:
 * transform b starts at element b * (number of points of one transform),
 * multi-dimensional transforms row-major (the last side contiguous).
 *
 * Ownership: the caller owns every buffer passed in.  A plan owns its
 * workspace and tables (allocated in fft_plan_create / fft_plan_create_nd,
 * freed in fft_plan_destroy).  polymul, polymul_batched and fft_convolve
 * allocate their scratch stream-ordered on the given stream and free it the
 * same way; polymul_noalloc uses a fixed device array of the library.
 *
 * Errors: every call returns FFT_OK (0) or one FFT_ERR_* code; calls that
 * return a pointer return NULL and record the code for fft_last_status()
 * (per host thread).  Arguments are validated before anything is enqueued;
 * FFT_ERR_CUDA means a CUDA runtime call or kernel launch failed, and
 * fft_last_cuda_error() names it.  Execution calls never synchronise the
 * device; plan creation may (it uploads or computes the plan's tables and
 * waits for them).
 */
#ifndef FFT_GB300_H
#define FFT_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define FFT_OK 0
#define FFT_ERR_INVALID_ARG 1 /* null pointer, size <= 0, bad enum value       */
#define FFT_ERR_NOT_POW2 2    /* kept for compatibility: no call returns it now */
#define FFT_ERR_UNSUPPORTED 3 /* valid but not implemented (size / dtype / dims) */
#define FFT_ERR_CUDA 4        /* CUDA runtime error or launch failure           */
#define FFT_ERR_ALLOC 5       /* device allocation failed                       */
#define FFT_ERR_MISALIGNED 6  /* a data pointer is not 16-byte aligned          */
#define FFT_ERR_DEVICE_TIMEOUT 7 /* a bounded wait inside a kernel ran out      */

/* Direction: the sign of the exponent. */
#define FFT_FORWARD (-1) /* e^{-i...}, unscaled          */
#define FFT_INVERSE (+1) /* e^{+i...}, scaled by 1/N     */

/* Element type. */
#define FFT_C2C_F32 0 /* interleaved float  (re, im), 8 bytes  */
#define FFT_C2C_F64 1 /* interleaved double (re, im), 16 bytes */
/* Transforms of real sequences (1D).  A real row of n samples has the
 * spectrum X_k = sum_j x_j e^{-2 pi i jk/n} with X_{n-k} = conj(X_k) ("FFT on
 * GPU", section Discrete Fourier Transform, for real x), so the half
 * spectrum X_0 .. X_{n/2} (n/2 + 1 bins, integer division) carries it all.
 *   FFT_FORWARD (R2C): in  = batch rows of n reals (float / double),
 *                      out = batch rows of n/2 + 1 interleaved complex bins.
 *   FFT_INVERSE (C2R): in  = batch rows of n/2 + 1 bins,
 *                      out = batch rows of n reals,
 *                      x_j = (1/n) sum_{k<n} Y_k e^{+2 pi i jk/n} with Y the
 *                      Hermitian extension (Y_k = X_k for k <= n/2,
 *                      conj(X_{n-k}) above); the imaginary parts of X_0 and
 *                      (even n) X_{n/2} are ignored.
 * Rows are contiguous with no padding (a row of bins starts every
 * (n/2 + 1) complex values).  Out of place only. */
#define FFT_REAL_F32 2 /* float samples, interleaved float bins   */
#define FFT_REAL_F64 3 /* double samples, interleaved double bins */

typedef struct fft_plan fft_plan;

/*
 * fft_plan_create -- plan `batch` transforms of length n (dims = 1) or of
 * n x n images (dims = 2) in the given direction and element type.
 *   n         1 <= n.  dims = 1: a power of two up to 2^30 (fp32) / 2^29
 *             (fp64), or any other length up to 2^26 (fp32) / 2^25 (fp64);
 *             batch * n * element size must fit the device.  dims = 2: as
 *             fft_plan_create_nd with shape {n, n}.
 *   batch     number of independent transforms, >= 1.
 *   dims      1, or 2 for an n x n transform (= fft_plan_create_nd with
 *             shape {n, n}).
 *   direction FFT_FORWARD or FFT_INVERSE.
 *   dtype     FFT_C2C_F32 or FFT_C2C_F64; or FFT_REAL_F32 / FFT_REAL_F64
 *             (dims = 1 only, else UNSUPPORTED) for real sequences, any
 *             n >= 1: n = 2H with H a power of two up to 2^14 (fp32) /
 *             2^13 (fp64) runs as one kernel per direction (the samples
 *             read as H complex values, a length-H transform on chip and
 *             the split into the half spectrum in the same block); other
 *             even n as a complex plan of length n/2 plus one kernel that
 *             splits or merges the spectrum over HBM (workspace batch * n/2
 *             complex); odd n as a complex plan of length n (workspace
 *             batch * n complex).
 * Lengths up to 2^14 (fp32) / 2^13 (fp64) run as one kernel in which one
 * thread block holds a whole transform on chip (one HBM read, one HBM write).
 * Longer 1D transforms run as 2-4 passes over HBM (a Stockham decomposition
 * into factors of at most 2^9) and need a workspace of batch * n elements,
 * allocated here on the current device.  Lengths that are not powers of two
 * ("FFT on GPU", sections FFT on GPU and Algorithm per signal Length): up to
 * 64 the direct DFT, one kernel; lengths whose only prime factors are 2, 3,
 * 5 and 7 up to 12288 (fp32) / 6144 (fp64) as mixed-radix Stockham stages
 * in one on-chip kernel; longer such lengths as N = N1 N2 (four-step: two
 * mixed-radix plans between three transposes, the middle one applying the
 * twiddles W_N^{n1 k2}; workspace batch * n); every other length by
 * Bluestein's algorithm -- a power-of-two convolution of length M >= 2n - 1
 * with a chirp -- whose chirp and filter spectrum are computed here (small
 * kernels on the legacy default stream, waited for) and kept by the plan,
 * plus 2 * batch * M work elements when M exceeds the on-chip length.
 * Returns NULL on error (fft_last_status(): INVALID_ARG, UNSUPPORTED, ALLOC,
 * CUDA).
 */
fft_plan *fft_plan_create(int64_t n, int64_t batch, int dims, int direction, int dtype);

/*
 * fft_plan_create_nd -- plan `batch` multi-dimensional transforms of shape
 * shape[0] x ... x shape[rank-1] (row-major: the last side is contiguous),
 * rank 1, 2 or 3 ("Stockham FFT Butterfly Algorithm in Parallel GLSL",
 * section Multi-Dimensional Transforms: the 1D transform along each axis in
 * turn, rows first).  Sides of any length 1 .. 2^30 (at most 2^40 elements
 * in all).  The inverse scales by 1/(product of the sides).  When every
 * side is a power of two, the last at most 2^14 (fp32) / 2^13 (fp64) and
 * the others at most the same, the plan is one on-chip row kernel plus one
 * in-place column pass per other axis, with no workspace -- except when
 * every side is 128 or 256: then each axis is one on-chip row kernel that
 * stores its output transposed (the next axis becomes contiguous), with a
 * workspace of batch * elements.  Otherwise the
 * contiguous axis runs as a 1D plan of any length (fft_plan_create), and
 * every other axis either as an in-place column pass (power-of-two length
 * and stride) or through a transpose into a workspace of batch * elements,
 * a 1D plan there, and a transpose back.  rank 1 is
 * fft_plan_create(shape[0], batch, 1, ...).  Errors as fft_plan_create.
 */
fft_plan *fft_plan_create_nd(int rank, const int64_t *shape, int64_t batch, int direction,
                             int dtype);

/* Frees the plan and its workspace.  NULL is ignored.  The caller must make
 * sure no fft_exec of this plan is still running on the GPU. */
void fft_plan_destroy(fft_plan *plan);

/* Bytes of device memory the plan owns (0 for single-kernel power-of-two
 * plans). */
size_t fft_plan_workspace_bytes(const fft_plan *plan);

/* Number of kernels one fft_exec of this plan launches. */
int fft_plan_num_kernels(const fft_plan *plan);

/*
 * fft_exec -- run the planned transforms.
 *   in, out   device pointers to batch-contiguous interleaved complex data
 *             of the plan's type (for FFT_REAL_* plans: reals and half
 *             spectra as described there), 16-byte aligned (else
 *             FFT_ERR_MISALIGNED).  in == out (in place) is allowed for
 *             complex plans (FFT_ERR_INVALID_ARG for real ones); other
 *             overlaps are not.  `in` is only read unless in == out.
 *   stream    a cudaStream_t (NULL = the legacy default stream).
 * Enqueues the kernels and returns; no synchronisation, no allocation, so
 * the call can be captured into a CUDA graph.  Plans that own a workspace
 * (fft_plan_workspace_bytes() > 0 beyond their tables: multi-pass,
 * Bluestein beyond the on-chip length, the split real kinds) use it on
 * every execution: executions of one such plan must not overlap on the GPU
 * (one stream, or events between streams); use one plan per concurrent
 * stream.
 */
int fft_exec(const fft_plan *plan, const void *in, void *out, void *stream);

/*
 * fft_exec_host -- fft_exec with host-side staging, all on `stream`:
 * if host_in is not NULL, copy host_in -> dev_in (cudaMemcpyAsync); run the
 * transform dev_in -> dev_out; if host_out is not NULL, copy
 * dev_out -> host_out.  Host buffers should be pinned for the copies to be
 * asynchronous.  dev_in / dev_out are caller-owned device buffers of the
 * plan's full input / output size (they may be equal for complex plans).
 * Allocates nothing.
 */
int fft_exec_host(const fft_plan *plan, const void *host_in, void *host_out, void *dev_in,
                  void *dev_out, void *stream);

/*
 * fft_exec_host_chain -- run plans[0], plans[1], ... plans[nplans-1] one
 * after the other on host data, streaming it through the device in chunks
 * of `chunk` transforms so that uploads, transforms and downloads of
 * different chunks overlap.  For each chunk: copy host_in -> dev_a, run
 * plans[0] dev_a -> dev_b, plans[1] dev_b -> dev_a, ..., copy the last
 * result (dev_a if nplans is even, dev_b if odd) -> host_out.
 *   plans     nplans >= 1 plans with the same batch, each taking as input
 *             what the previous one produces (same bytes per transform:
 *             e.g. an R2C plan followed by the C2R plan of the same n).
 *   host_in, host_out  host buffers of the full batch (pinned for the copies
 *             to overlap); host_in is only read.
 *   dev_a, dev_b       caller-owned device buffers, each large enough for
 *             the full batch of every input or output placed in it,
 *             16-byte aligned; both are overwritten; distinct when a real
 *             plan is in the chain (else FFT_ERR_INVALID_ARG).
 *   chunk     transforms per chunk (>= 1; at most 4096 chunks); every
 *             chunk's slice of every buffer must start 16-byte aligned
 *             (else FFT_ERR_MISALIGNED).
 * Ordered after the work already on `stream`; `stream` waits for the last
 * download, so the call is asynchronous on `stream` like fft_exec.  Uses
 * three internal non-blocking streams and per-chunk events, created on the
 * first call on a device (calls on one device are serialised by a lock
 * while they enqueue).  Allocates no device memory.
 */
int fft_exec_host_chain(const fft_plan *const *plans, int nplans, const void *host_in,
                        void *host_out, void *dev_a, void *dev_b, int64_t chunk, void *stream);

/*
 * polymul -- c = a * b for integer coefficient vectors (device pointers,
 * int64, 8-byte aligned): a has na >= 1 coefficients, b has nb >= 1,
 * c receives na + nb - 1.  The product is formed with fp64 transforms of
 * length L = the smallest power of two >= na + nb - 1 (zero padding), the
 * pointwise product of the two spectra, the inverse transform, and rounding
 * to the nearest integer.  The result is exact while every |c_k| and the
 * transform's rounding error stay well below 2^52 and 0.5 respectively
 * (e.g. coefficients in [0, 9] with na, nb <= 2^20 give |c_k| < 2^27 and an
 * error of order 1e-7).  L <= 2^27.  Both inputs ride in one complex
 * transform (a + i b) and the real product comes back through one of length
 * L/2.  Scratch of 2 * L * 16 bytes plus six twiddle tables of
 * 2^ceil(log2(L) / 2) complex doubles each (6 * 16 * 2^ceil(log2(L) / 2)
 * bytes: 192 KiB at L = 2^21, 1.5 MiB at L = 2^27) is allocated with
 * cudaMallocAsync on `stream` and freed the same way.
 */
int polymul(const int64_t *a, int64_t na, const int64_t *b, int64_t nb, int64_t *c,
            void *stream);

/* Number of kernels one polymul / polymul_batched / polymul_noalloc call
 * with these lengths launches (0 if the lengths are invalid). */
int polymul_num_kernels(int64_t na, int64_t nb);

/* polymul over `batch` independent pairs: pair p uses a + p*na, b + p*nb
 * and writes c + p*(na+nb-1).  Scratch is 2 * batch * L * 16 bytes plus
 * the same six twiddle tables as polymul's. */
int polymul_batched(const int64_t *a, int64_t na, const int64_t *b, int64_t nb, int64_t *c,
                    int64_t batch, void *stream);

/*
 * polymul_batched_host -- polymul_batched of coefficient arrays in host
 * memory, streamed through the device in chunks of `chunk` pairs: for each
 * chunk its rows of a_host and b_host are copied to dev_a / dev_b, multiplied
 * into dev_c (polymul_batched on that range) and copied back to c_host,
 * overlapping across chunks on three internal streams.
 *   a_host, b_host, c_host  host arrays of batch * na, batch * nb and
 *             batch * (na + nb - 1) int64 (pinned for the copies to overlap).
 *   dev_a, dev_b, dev_c     caller-owned device arrays of the same sizes,
 *             8-byte aligned.
 *   chunk     pairs per chunk (>= 1; at most 4096 chunks).
 * Errors as polymul_batched; asynchronous on `stream`.
 */
int polymul_batched_host(const int64_t *a_host, int64_t na, const int64_t *b_host, int64_t nb,
                         int64_t *c_host, int64_t batch, int64_t *dev_a, int64_t *dev_b,
                         int64_t *dev_c, int64_t chunk, void *stream);

/*
 * polymul_noalloc -- the same product as polymul for one pair, for callers
 * that must not allocate device memory where they need it (a plug-in whose
 * host application owns the device-memory budget, or a latency-critical
 * loop where an allocation could wait on the device or fail).  The source
 * pages have no counterpart: this is a property of this library's memory
 * handling, not of the method.
 *   a, b, c  as for polymul (device pointers, int64, 8-byte aligned).
 *   na + nb - 1 must be at most FFT_POLYMUL_NOALLOC_MAX_LEN; longer products
 *            return FFT_ERR_UNSUPPORTED (use polymul for them).
 * Scratch: a fixed 3 MiB array in the library's device image (every GPU that
 * loads the library holds it until the process exits).  No call allocates
 * or frees memory.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current -- make that
 * first call outside any stream capture.  cudaDeviceReset destroys the
 * array with the device's context; the first call after it looks the
 * address up again in the new context (make that call outside any capture
 * too).  All calls on a device share the array: calls that overlap on the
 * GPU race and give wrong results, so order them on one stream.  Nothing in
 * the array needs clearing between calls.
 */
#define FFT_POLYMUL_NOALLOC_MAX_LEN 65536
int polymul_noalloc(const int64_t *a, int64_t na, const int64_t *b, int64_t nb, int64_t *c,
                    void *stream);

/* Sample types of fft_convolve. */
#define FFT_CONV_COMPLEX 0 /* interleaved complex samples of dtype */
#define FFT_CONV_REAL 1    /* real samples: float (FFT_C2C_F32) or double (FFT_C2C_F64) */

/*
 * fft_convolve -- linear convolution of every row of x with a filter:
 *   y[b][k] = sum_i x[b][i] h[k-i],  k < nx + nh - 1
 * (the coefficient convolution of "FFT on GPU", polynomial-multiplication
 * section, for complex or real samples), computed as the inverse transform
 * of the pointwise product of the zero-padded forward transforms, length
 * L = the smallest power of two >= nx + nh - 1.
 *   x         device pointer, batch rows of nx samples (row-major).
 *   h         device pointer: nh samples (h_per_row = 0, one filter for every
 *             row) or batch rows of nh samples (h_per_row = 1).
 *   y         device pointer, batch rows of nx + nh - 1 samples (written).
 *   kind      FFT_CONV_COMPLEX or FFT_CONV_REAL; dtype FFT_C2C_F32 / _F64.
 *             Pointers aligned to their sample size (else MISALIGNED).
 * L <= 2^14 (fp32) / 2^13 (fp64): each row is read once and written once
 * by one kernel (transform, product, inverse on chip).  Longer: 2-4 HBM
 * passes per transform.  Real rows with one shared filter are transformed
 * two at a time (as the real and imaginary parts of one complex signal).
 * L <= 2^27 (fp32) / 2^26 (fp64).  Scratch (the filter spectra, and for long
 * transforms two work arrays) is allocated with cudaMallocAsync on `stream`
 * and freed the same way.  Asynchronous on `stream`.
 */
int fft_convolve(const void *x, int64_t nx, const void *h, int64_t nh, void *y, int64_t batch,
                 int h_per_row, int kind, int dtype, void *stream);

/* Kernels one fft_convolve call with these arguments launches (0 if the
 * arguments are invalid). */
int fft_convolve_num_kernels(int64_t nx, int64_t nh, int64_t batch, int h_per_row, int kind,
                             int dtype);

/*
 * fft_convolve_host -- fft_convolve of signals in host memory, streamed
 * through the device in chunks of `chunk` rows: for each chunk the rows of
 * x_host are copied to dev_x, convolved into dev_y (fft_convolve on that
 * range of rows) and copied back to y_host, uploads, convolutions and
 * downloads of different chunks overlapping on three internal streams
 * (as fft_exec_host_chain).
 *   x_host, y_host  host buffers of batch * nx and batch * (nx + nh - 1)
 *             samples (pinned for the copies to overlap); x_host only read.
 *   h         DEVICE pointer to the filter(s), as for fft_convolve.
 *   dev_x, dev_y    caller-owned device buffers of the same full sizes.
 *   chunk     rows per chunk (>= 1; at most 4096 chunks).
 * Other arguments and errors as fft_convolve; asynchronous on `stream`.
 */
int fft_convolve_host(const void *x_host, int64_t nx, const void *h, int64_t nh, void *y_host,
                      int64_t batch, int h_per_row, int kind, int dtype, void *dev_x, void *dev_y,
                      int64_t chunk, void *stream);

/*
 * fft_debug_radix2_pass -- test hook (not part of the transform API): one
 * gather-shaped radix-2 butterfly pass, "The Butterfly: One Thread, One
 * Output" (gpu.rocks FFT butterfly, task 2).  Output cell i takes
 * j = floor(i/half) mod 2, base = i - j*half, r = i mod half,
 * a = in[base], b = in[base+half], w = e^{-i pi r / half} and writes
 * a + w b (j = 0) or a - w b (j = 1).
 *   in, out  device pointers, n interleaved complex values of `dtype`;
 *            must not overlap.
 *   n        > 0, a multiple of 2*half;  half >= 1.
 */
int fft_debug_radix2_pass(const void *in, void *out, int64_t n, int64_t half, int dtype,
                          void *stream);

/*
 * fft_device_status -- synchronises `stream`, then reads and clears the
 * library's device status word on the current device.  Kernels that wait
 * for their own asynchronous copies (the TMA-staged HBM passes) bound every
 * wait; a wait that runs out sets the word and the kernel stops early, so
 * its output is incomplete.  Returns FFT_OK, FFT_ERR_DEVICE_TIMEOUT, or
 * FFT_ERR_CUDA if the synchronisation itself failed.  Diagnostic: no
 * transform call reads the word by itself.
 */
int fft_device_status(void *stream);

/*
 * fft_debug_wait_timeout -- test hook (not part of the transform API): one
 * block waits on an mbarrier transaction that never arrives, `polls` times
 * (1 .. 2^22), and records the timeout in the device status word exactly as
 * the TMA pass kernel does; fft_device_status then reports
 * FFT_ERR_DEVICE_TIMEOUT.  Issues no copy and faults nothing.  No
 * counterpart on the source pages.
 */
int fft_debug_wait_timeout(int64_t polls, void *stream);

/*
 * fft_debug_cluster_timeout -- test hook (not part of the transform API):
 * runs the cluster pass kernel once, in place, on `data` (device, 16-byte
 * aligned, 2^15 fp32 complex values = 256 KiB, overwritten with
 * meaningless values), with the tile load of one of its 8 blocks armed for
 * 16 bytes that never arrive and every load wait bounded to `polls` polls
 * (1 .. 2^22).  That block's wait runs out; the whole cluster sees its
 * flag, leaves together, and the device status word reads
 * FFT_ERR_DEVICE_TIMEOUT (fft_device_status).  Returns FFT_ERR_UNSUPPORTED
 * when the cluster kernel is switched off (FFT_OPT_NO_CLUSTER).  Faults
 * nothing.  No counterpart on the source pages.
 */
int fft_debug_cluster_timeout(void *data, int64_t polls, void *stream);

/*
 * fft_debug_set_option -- test and tuning hook (not part of the transform
 * API; no transform needs it): sets one process-wide choice that the
 * planner and the pass launchers otherwise make themselves, so that tests
 * can run every schedule on small shapes and kernels can be compared.  A
 * plan reads the planning options when it is created; the launch options
 * apply to every later launch.  `value` < 0 restores the library's own
 * choice.  Nothing in the library reads the process environment.  Returns
 * FFT_OK, or FFT_ERR_INVALID_ARG for an unknown option or a value out of
 * its range (the option is then unchanged).  Not thread-safe with respect
 * to plans being created or launched at the same time.
 */
#define FFT_OPT_PASS_LOG 1        /* planning: largest on-chip factor (log2, 4 .. 14 fp32,
                                     4 .. 13 fp64) per HBM pass of a long 1D transform;
                                     own choice 9 */
#define FFT_OPT_PASS_SPLIT 2      /* planning: the passes of a long 1D transform, one factor
                                     (log2, 1 .. 14) per 4 bits, first pass in the lowest;
                                     used when they add up to log2 N */
#define FFT_OPT_NO_TMA 3          /* launch: 1 = every pass by the plain-load kernel */
#define FFT_OPT_NO_CLUSTER 4      /* launch: 1 = no thread-block-cluster passes */
#define FFT_OPT_CLUSTER_LOG_MIN 5 /* launch: shortest on-chip length (log2, 11 .. 13) that
                                     takes the cluster pass; own choice 12 */
#define FFT_OPT_ND_ROWS_T 6       /* planning: 2D / 3D of power-of-two sides as rows with
                                     transposed stores (1) or rows + column passes (0);
                                     own choice by shape */
#define FFT_OPT_COL_RADIX_LOG 7   /* planning: 2D / 3D, out of place: log2 of the radix of the
                                     column transform's first stage folded into the row pass
                                     (0 = none, 1 .. 3); own choice log2(H / 512) for columns
                                     of 1024 and 2048 points (blocks of at most 512 threads),
                                     2 (1 for rows of 4096 points) for 4096 and 8192 */
#define FFT_OPT_ROWS_SHFL 8       /* launch: 1 = 512-point on-chip transforms exchange data
                                     between stages by warp shuffles (one warp per transform)
                                     instead of shared memory; own choice 0 */
#define FFT_OPT_PASS_SHFL 9       /* launch: 1 = fp32 HBM passes of 512-point columns give each
                                     column to one warp and exchange by warp shuffles (tiles
                                     loaded and stored with the TMA's 64-byte swizzle);
                                     0 = shared-memory exchanges */
int fft_debug_set_option(int option, int64_t value);

/* Last status recorded on this host thread by a call that returns a
 * pointer (fft_plan_create). */
int fft_last_status(void);

/* Static description of a status code. */
const char *fft_status_string(int status);

/* Name of the last CUDA error seen by this library on this host thread
 * ("no error" if none). */
const char *fft_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FFT_GB300_H */
