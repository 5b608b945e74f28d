/*
 * fft_oracle.c -- plain, slow, obviously-correct fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link, call or execute this file.  It
 * exists so that tests, the smoke check and the CPU baseline of the bench
 * have an independent answer to compare against.  It shares no code, table
 * or constant with the GPU path.
 *
 * Every routine is a direct transcription of a definition on the source
 * pages, written for readability, not speed:
 *
 *   "FFT on GPU" (elwhyjay.github.io/post/fft)
 *     - Discrete Fourier Transform: X_k = sum_n x_n e^{-i 2 pi k n / N}
 *     - Primitive Root of Unity: omega_N = e^{-i 2 pi / N}
 *     - Fast Fourier Transform: even/odd split, X_k = E_k + omega^k O_k,
 *       X_{k+N/2} = E_k - omega^k O_k
 *     - polynomial multiplication: coefficient convolution
 *       c_k = sum_i a_i b_{k-i}; inverse a_j = (1/N) sum_k A_k omega^{-jk}
 *     - reverse bit order: the 8-point order [x0,x4,x2,x6,x1,x5,x3,x7]
 *     - the same coefficient convolution written for complex sequences is
 *       the linear convolution of signals: y_k = sum_i x_i h_{k-i}
 *   "The Butterfly: One Thread, One Output" (gpu.rocks, FFT butterfly task 2)
 *     - one gather-shaped radix-2 pass: j = floor(i/half) mod 2,
 *       base = i - j*half, r = i mod half, w = e^{-i pi r / half}
 *   "Stockham FFT Butterfly Algorithm in Parallel GLSL" (salivity.github.io)
 *     - one Stockham stage s: j = floor(x/2^{s+1}) 2^s + (x mod 2^s),
 *       k = j + N/2, r = (x mod 2^{s+1}) N / 2^{s+1}.  The page does not
 *       write the combine step; it is read here as
 *       out[x] = in[j] + W_N^r in[k]  (W_N^r = e^{-i 2 pi r / N}).
 *
 * Data layout of every complex array: interleaved (re, im) doubles, the
 * layout of the pages' CUDA code (signal[2*i], signal[2*i+1]).
 *
 * Sign convention: sign = -1 is the forward transform (e^{-i...}, unscaled),
 * sign = +1 the inverse kernel (e^{+i...}); the "inverse" entry points also
 * apply the 1/N factor of the inverse formula.
 *
 * Every entry point returns 0 on success and a negative number on bad
 * arguments.
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef double _Complex cplx;

static const double TWO_PI = 6.28318530717958647692528676655900577;

static int is_pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }

/* (a * b) mod n for 0 <= a, b < n, without overflow. */
static int64_t mulmod(int64_t a, int64_t b, int64_t n) {
    return (int64_t)(((unsigned __int128)a * (unsigned __int128)b) % (unsigned __int128)n);
}

/* omega_N^m with omega_N = e^{sign i 2 pi / N}; m is first reduced mod N in
 * integers so that the angle is always in [0, 2 pi). */
static cplx root_of_unity(int64_t m, int64_t n, int sign) {
    int64_t r = m % n;
    if (r < 0) r += n;
    double ang = TWO_PI * (double)r / (double)n;
    return cos(ang) + (double)sign * sin(ang) * I;
}

/* Exposed so the tests can check the root-of-unity identities
 * (periodicity, omega^{k+N/2} = -omega^k, omega_N^{2k} = omega_{N/2}^k). */
int oracle_root_of_unity(int64_t m, int64_t n, int sign, double *out2) {
    if (n <= 0 || out2 == NULL || (sign != 1 && sign != -1)) return -1;
    cplx w = root_of_unity(m, n, sign);
    out2[0] = creal(w);
    out2[1] = cimag(w);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Direct DFT, O(N^2): X_k = sum_n x_n omega_N^{kn}.  The exponent k*n is
 * reduced mod N exactly; the sum is Kahan-compensated on each component.
 * Any N >= 1 (the definition needs no power of two).
 * ------------------------------------------------------------------------- */
static cplx dft_one_bin(const cplx *x, int64_t n, int sign, int64_t k) {
    double sr = 0.0, si = 0.0, cr = 0.0, ci = 0.0;
    int64_t kk = k % n;
    if (kk < 0) kk += n;
    for (int64_t j = 0; j < n; ++j) {
        cplx term = x[j] * root_of_unity(mulmod(kk, j, n), n, sign);
        double yr = creal(term) - cr;
        double tr = sr + yr;
        cr = (tr - sr) - yr;
        sr = tr;
        double yi = cimag(term) - ci;
        double ti = si + yi;
        ci = (ti - si) - yi;
        si = ti;
    }
    return sr + si * I;
}

int oracle_dft(const double *x, int64_t n, int sign, double *X) {
    if (n <= 0 || x == NULL || X == NULL || (sign != 1 && sign != -1)) return -1;
    const cplx *xc = (const cplx *)x;
    cplx *out = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    if (!out) return -2;
    for (int64_t k = 0; k < n; ++k) out[k] = dft_one_bin(xc, n, sign, k);
    memcpy(X, out, sizeof(cplx) * (size_t)n);
    free(out);
    return 0;
}

/* Selected bins only: X[t] = X_{ks[t]}, O(N) per bin (for large N). */
int oracle_dft_bins(const double *x, int64_t n, int sign, const int64_t *ks, int64_t nk,
                    double *X) {
    if (n <= 0 || x == NULL || X == NULL || ks == NULL || nk < 0 ||
        (sign != 1 && sign != -1))
        return -1;
    const cplx *xc = (const cplx *)x;
    cplx *out = (cplx *)X;
    for (int64_t t = 0; t < nk; ++t) out[t] = dft_one_bin(xc, n, sign, ks[t]);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Recursive even/odd Cooley-Tukey, exactly the derivation on the page:
 *   E = DFT_{N/2}(x_0, x_2, ...),  O = DFT_{N/2}(x_1, x_3, ...)
 *   X_k = E_k + omega_N^k O_k,  X_{k+N/2} = E_k - omega_N^k O_k.
 * The two half-length results are computed into the two halves of the
 * output, which the combine loop then overwrites pairwise.  omega_N^k is
 * evaluated directly from cos/sin at every level (never by repeated
 * multiplication).  N must be a power of two.
 * ------------------------------------------------------------------------- */
static void ct_recursive(const cplx *x, int64_t stride, int64_t n, int sign, cplx *X) {
    if (n == 1) {
        X[0] = x[0];
        return;
    }
    int64_t h = n / 2;
    ct_recursive(x, 2 * stride, h, sign, X);          /* E_k into X[0..h)  */
    ct_recursive(x + stride, 2 * stride, h, sign, X + h); /* O_k into X[h..n) */
    for (int64_t k = 0; k < h; ++k) {
        cplx e = X[k];
        cplx o = root_of_unity(k, n, sign) * X[k + h];
        X[k] = e + o;
        X[k + h] = e - o;
    }
}

int oracle_fft(const double *x, int64_t n, int sign, double *X) {
    if (!is_pow2(n) || x == NULL || X == NULL || (sign != 1 && sign != -1)) return -1;
    cplx *out = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    if (!out) return -2;
    ct_recursive((const cplx *)x, 1, n, sign, out);
    memcpy(X, out, sizeof(cplx) * (size_t)n);
    free(out);
    return 0;
}

/* Inverse transform: conjugate root (sign +1) and the factor 1/N. */
int oracle_ifft(const double *X, int64_t n, double *x) {
    int rc = oracle_fft(X, n, +1, x);
    if (rc) return rc;
    double s = 1.0 / (double)n;
    for (int64_t i = 0; i < 2 * n; ++i) x[i] *= s;
    return 0;
}

int oracle_idft(const double *X, int64_t n, double *x) {
    int rc = oracle_dft(X, n, +1, x);
    if (rc) return rc;
    double s = 1.0 / (double)n;
    for (int64_t i = 0; i < 2 * n; ++i) x[i] *= s;
    return 0;
}

/* Batched forms: `batch` transforms of length n, contiguous, stride n.
 * direction -1 = forward, +1 = inverse with 1/N. */
int oracle_fft_batch(const double *x, int64_t n, int64_t batch, int direction, double *X) {
    if (batch < 0) return -1;
    for (int64_t b = 0; b < batch; ++b) {
        int rc = direction < 0 ? oracle_fft(x + 2 * n * b, n, -1, X + 2 * n * b)
                               : oracle_ifft(x + 2 * n * b, n, X + 2 * n * b);
        if (rc) return rc;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Separable 2D transform of one h x w row-major image: 1D transforms along
 * every row (the contiguous axis), then along every column.  direction -1
 * forward, +1 inverse (1/(h*w) in total, 1/w from the rows, 1/h from the
 * columns).
 * ------------------------------------------------------------------------- */
int oracle_fft2d(const double *x, int64_t h, int64_t w, int direction, double *X) {
    if (!is_pow2(h) || !is_pow2(w) || x == NULL || X == NULL) return -1;
    cplx *img = (cplx *)malloc(sizeof(cplx) * (size_t)(h * w));
    cplx *col = (cplx *)malloc(sizeof(cplx) * (size_t)h);
    cplx *tmp = (cplx *)malloc(sizeof(cplx) * (size_t)(h > w ? h : w));
    if (!img || !col || !tmp) {
        free(img); free(col); free(tmp);
        return -2;
    }
    int sign = direction < 0 ? -1 : +1;
    const cplx *xc = (const cplx *)x;
    for (int64_t r = 0; r < h; ++r) {
        ct_recursive(xc + r * w, 1, w, sign, tmp);
        for (int64_t c = 0; c < w; ++c) img[r * w + c] = tmp[c];
    }
    for (int64_t c = 0; c < w; ++c) {
        for (int64_t r = 0; r < h; ++r) col[r] = img[r * w + c];
        ct_recursive(col, 1, h, sign, tmp);
        for (int64_t r = 0; r < h; ++r) img[r * w + c] = tmp[r];
    }
    double s = direction < 0 ? 1.0 : 1.0 / ((double)h * (double)w);
    cplx *out = (cplx *)X;
    for (int64_t i = 0; i < h * w; ++i) out[i] = img[i] * s;
    free(img); free(col); free(tmp);
    return 0;
}

/* ---------------------------------------------------------------------------
 * One gather-shaped radix-2 pass (gpu.rocks butterfly task 2): every output
 * cell i reads its own pair and twiddle and writes only itself.
 * n must be a multiple of 2*half.
 * ------------------------------------------------------------------------- */
int oracle_radix2_pass(const double *x, int64_t n, int64_t half, double *y) {
    if (half <= 0 || n <= 0 || n % (2 * half) != 0 || x == NULL || y == NULL) return -1;
    const cplx *xc = (const cplx *)x;
    cplx *out = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    if (!out) return -2;
    for (int64_t i = 0; i < n; ++i) {
        int64_t j = (i / half) % 2;      /* 0 = lower member, 1 = upper */
        int64_t base = i - j * half;     /* the lower member's index    */
        int64_t r = i % half;            /* position in the half-block  */
        cplx a = xc[base];
        cplx b = xc[base + half];
        /* w = e^{-i pi r / half} = omega_{2 half}^r */
        cplx wb = root_of_unity(r, 2 * half, -1) * b;
        out[i] = (j == 0) ? a + wb : a - wb;
    }
    memcpy(y, out, sizeof(cplx) * (size_t)n);
    free(out);
    return 0;
}

/* Bit-reversal permutation: y[i] = x[rev(i)] over log2(n) bits. */
int oracle_bit_reverse(const double *x, int64_t n, double *y) {
    if (!is_pow2(n) || x == NULL || y == NULL) return -1;
    int bits = 0;
    while (((int64_t)1 << bits) < n) ++bits;
    const cplx *xc = (const cplx *)x;
    cplx *out = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    if (!out) return -2;
    for (int64_t i = 0; i < n; ++i) {
        int64_t rev = 0, t = i;
        for (int b = 0; b < bits; ++b) {
            rev = (rev << 1) | (t & 1);
            t >>= 1;
        }
        out[i] = xc[rev];
    }
    memcpy(y, out, sizeof(cplx) * (size_t)n);
    free(out);
    return 0;
}

/* Exposed for the golden check of the printed 8-point order. */
int oracle_bit_reverse_index(int64_t i, int64_t n, int64_t *rev_out) {
    if (!is_pow2(n) || i < 0 || i >= n || rev_out == NULL) return -1;
    int bits = 0;
    while (((int64_t)1 << bits) < n) ++bits;
    int64_t rev = 0, t = i;
    for (int b = 0; b < bits; ++b) {
        rev = (rev << 1) | (t & 1);
        t >>= 1;
    }
    *rev_out = rev;
    return 0;
}

/* One Stockham autosort stage s in [0, log2 n), forward sign. */
int oracle_stockham_stage(const double *x, int64_t n, int s, double *y) {
    if (!is_pow2(n) || n < 2 || s < 0 || ((int64_t)1 << (s + 1)) > n || x == NULL || y == NULL)
        return -1;
    const cplx *xc = (const cplx *)x;
    cplx *out = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    if (!out) return -2;
    int64_t span = (int64_t)1 << (s + 1); /* 2^{s+1} */
    int64_t half = (int64_t)1 << s;       /* 2^s     */
    for (int64_t xi = 0; xi < n; ++xi) {
        int64_t j = (xi / span) * half + (xi % half);
        int64_t k = j + n / 2;
        int64_t r = (xi % span) * (n / span);
        out[xi] = xc[j] + root_of_unity(r, n, -1) * xc[k];
    }
    memcpy(y, out, sizeof(cplx) * (size_t)n);
    free(out);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Polynomial multiplication.
 * ------------------------------------------------------------------------- */

/* Coefficient form, schoolbook: c_k = sum_{i} a_i b_{k-i}, at the requested
 * output indices only (each O(min(na, nb))).  Accumulates in 128-bit
 * integers; returns -3 if a result does not fit in int64. */
int oracle_polymul_schoolbook_at(const int64_t *a, int64_t na, const int64_t *b, int64_t nb,
                                 const int64_t *idx, int64_t nidx, int64_t *c) {
    if (na <= 0 || nb <= 0 || a == NULL || b == NULL || idx == NULL || c == NULL || nidx < 0)
        return -1;
    for (int64_t t = 0; t < nidx; ++t) {
        int64_t k = idx[t];
        if (k < 0 || k > na + nb - 2) return -1;
        int64_t lo = k - (nb - 1) > 0 ? k - (nb - 1) : 0;
        int64_t hi = k < na - 1 ? k : na - 1;
        __int128 s = 0;
        for (int64_t i = lo; i <= hi; ++i) s += (__int128)a[i] * (__int128)b[k - i];
        if (s > (__int128)INT64_MAX || s < (__int128)INT64_MIN) return -3;
        c[t] = (int64_t)s;
    }
    return 0;
}

/* The full transform pipeline in fp64: zero-pad both coefficient vectors to
 * L = the smallest power of two >= na+nb-1, forward transform both, multiply
 * pointwise (point-value form), inverse transform with 1/L, round each real
 * part to the nearest integer.  Writes na+nb-1 coefficients. */
int oracle_polymul_fft(const int64_t *a, int64_t na, const int64_t *b, int64_t nb, int64_t *c) {
    if (na <= 0 || nb <= 0 || a == NULL || b == NULL || c == NULL) return -1;
    int64_t nc = na + nb - 1;
    int64_t L = 1;
    while (L < nc) L <<= 1;
    cplx *pa = (cplx *)calloc((size_t)L, sizeof(cplx));
    cplx *pb = (cplx *)calloc((size_t)L, sizeof(cplx));
    cplx *A = (cplx *)malloc(sizeof(cplx) * (size_t)L);
    cplx *B = (cplx *)malloc(sizeof(cplx) * (size_t)L);
    if (!pa || !pb || !A || !B) {
        free(pa); free(pb); free(A); free(B);
        return -2;
    }
    for (int64_t i = 0; i < na; ++i) pa[i] = (double)a[i];
    for (int64_t i = 0; i < nb; ++i) pb[i] = (double)b[i];
    ct_recursive(pa, 1, L, -1, A);
    ct_recursive(pb, 1, L, -1, B);
    for (int64_t k = 0; k < L; ++k) A[k] = A[k] * B[k];
    ct_recursive(A, 1, L, +1, pa);
    for (int64_t k = 0; k < nc; ++k) c[k] = llround(creal(pa[k]) / (double)L);
    free(pa); free(pb); free(A); free(B);
    return 0;
}

/* P(t) mod p by Horner's rule, p = 2^61 - 1 (a prime), for the
 * point-value identity C(t) = A(t) B(t) checked modulo p. */
int oracle_poly_eval_mod(const int64_t *a, int64_t na, uint64_t t, uint64_t *out) {
    const uint64_t p = ((uint64_t)1 << 61) - 1;
    if (na < 0 || (na > 0 && a == NULL) || out == NULL) return -1;
    uint64_t tt = t % p;
    unsigned __int128 acc = 0;
    for (int64_t i = na - 1; i >= 0; --i) {
        int64_t ai = a[i];
        uint64_t ar = ai >= 0 ? (uint64_t)ai % p : (p - ((uint64_t)(-(ai + 1)) + 1) % p) % p;
        acc = (acc * tt + ar) % p;
    }
    *out = (uint64_t)acc;
    return 0;
}

/* ---------------------------------------------------------------------------
 * Linear convolution of complex sequences, the definition written out:
 *   y_k = sum_i x_i h_{k-i},  k = 0 .. nx+nh-2,
 * Kahan-compensated on each component.  O(nx * nh).
 * ------------------------------------------------------------------------- */
int oracle_convolve(const double *x, int64_t nx, const double *h, int64_t nh, double *y) {
    if (nx <= 0 || nh <= 0 || x == NULL || h == NULL || y == NULL) return -1;
    const cplx *xc = (const cplx *)x;
    const cplx *hc = (const cplx *)h;
    cplx *out = (cplx *)y;
    for (int64_t k = 0; k < nx + nh - 1; ++k) {
        int64_t lo = k - (nh - 1) > 0 ? k - (nh - 1) : 0;
        int64_t hi = k < nx - 1 ? k : nx - 1;
        double sr = 0.0, si = 0.0, cr = 0.0, ci = 0.0;
        for (int64_t i = lo; i <= hi; ++i) {
            cplx term = xc[i] * hc[k - i];
            double yr = creal(term) - cr;
            double tr = sr + yr;
            cr = (tr - sr) - yr;
            sr = tr;
            double yi = cimag(term) - ci;
            double ti = si + yi;
            ci = (ti - si) - yi;
            si = ti;
        }
        out[k] = sr + si * I;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Transforms of real sequences.  For real x the DFT X_k = sum_n x_n omega^{kn}
 * satisfies X_{N-k} = conj(X_k), so the bins k = 0 .. floor(N/2) hold all of
 * it (the half spectrum).
 *
 *   oracle_rfft:  X_k, k = 0 .. floor(N/2), of the DFT of x_n + 0i
 *                 (forward, unscaled).  x: n doubles; X: floor(n/2)+1 complex.
 *   oracle_irfft: the inverse of a half spectrum: the full spectrum
 *                 Y_k = X_k (k <= N/2), Y_k = conj(X_{N-k}) (k > N/2), its
 *                 inverse transform with 1/N, and the real part of that.  The
 *                 imaginary parts of X_0 and (even N) X_{N/2} add only
 *                 imaginary terms to the result and so drop out.
 *                 X: floor(n/2)+1 complex; x: n doubles.
 * Power-of-two N goes through the recursive Cooley-Tukey, every other N
 * through the direct DFT.
 * ------------------------------------------------------------------------- */
static int full_transform(const cplx *x, int64_t n, int sign, cplx *X) {
    return is_pow2(n) ? oracle_fft((const double *)x, n, sign, (double *)X)
                      : oracle_dft((const double *)x, n, sign, (double *)X);
}

int oracle_rfft(const double *x, int64_t n, double *X) {
    if (n <= 0 || x == NULL || X == NULL) return -1;
    cplx *z = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    cplx *Z = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    if (!z || !Z) {
        free(z); free(Z);
        return -2;
    }
    for (int64_t i = 0; i < n; ++i) z[i] = x[i] + 0.0 * I;
    int rc = full_transform(z, n, -1, Z);
    if (rc == 0) memcpy(X, Z, sizeof(cplx) * (size_t)(n / 2 + 1));
    free(z);
    free(Z);
    return rc;
}

int oracle_irfft(const double *X, int64_t n, double *x) {
    if (n <= 0 || x == NULL || X == NULL) return -1;
    const cplx *half = (const cplx *)X;
    cplx *Y = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    cplx *y = (cplx *)malloc(sizeof(cplx) * (size_t)n);
    if (!Y || !y) {
        free(Y); free(y);
        return -2;
    }
    for (int64_t k = 0; k < n; ++k) Y[k] = 2 * k <= n ? half[k] : conj(half[n - k]);
    int rc = full_transform(Y, n, +1, y);
    if (rc == 0)
        for (int64_t i = 0; i < n; ++i) x[i] = creal(y[i]) / (double)n;
    free(Y);
    free(y);
    return rc;
}
