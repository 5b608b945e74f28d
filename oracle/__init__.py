"""fp64 CPU oracle for the power-of-two FFT, the 2D FFT and FFT polynomial
multiplication.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``fft_convolution_gb300``) never imports, links or runs it, and
this package imports nothing from the product path: the two share no code.

The arithmetic lives in ``fft_oracle.c`` (plain C, fp64, libm cos/sin); this
module only builds it with gcc, loads it with ctypes and marshals numpy
arrays.  Every function states the passage it follows:

* ``dft`` / ``dft_bins`` -- the DFT definition, "FFT on GPU", section
  Discrete Fourier Transform (X_k = sum_n x_n e^{-i 2 pi k n / N}).
* ``fft`` / ``ifft`` -- the recursive even/odd Cooley-Tukey derivation,
  "FFT on GPU", section Fast Fourier Transform; the inverse with the conjugate
  root and 1/N, section "polynomial multiplication and FFT".
* ``fft2d`` / ``fftn`` -- separable 2D / nD: rows, then columns (then depth),
  "Stockham FFT Butterfly Algorithm in Parallel GLSL", section
  Multi-Dimensional Transforms.
* ``radix2_pass`` -- one gather-shaped pass, "The Butterfly: One Thread, One
  Output" (gpu.rocks), the j / base / r recipe.
* ``stockham_stage`` -- one Stockham stage, "Stockham FFT Butterfly Algorithm
  in Parallel GLSL", section Execution via GLSL Compute Shaders, items 2-3.
* ``bit_reverse`` -- "FFT on GPU", section reverse bit order.
* ``polymul_*`` / ``poly_eval_mod`` -- "FFT on GPU", sections on the two
  representations of a polynomial and the whole pipeline.
* ``convolve`` -- the same coefficient convolution c_k = sum_i a_i b_{k-i}
  for complex signals (linear convolution), summed directly.

Every oracle function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle.py`` to something other than itself (closed forms,
printed values, invariants, numpy's FFT, exact big-integer arithmetic).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fft_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_U64 = ctypes.POINTER(ctypes.c_uint64)


def build(force: bool = False) -> str:
    """Compile fft_oracle.c into liboracle.so next to it (gcc, -O2, IEEE
    arithmetic: no fast-math).  Returns the library path."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(lib):
    """Set the ctypes signatures of every oracle entry point on `lib` (a
    CDLL of fft_oracle.c, or of a deliberately mutated copy in the pin
    tests)."""
    i64, c_int = ctypes.c_int64, ctypes.c_int
    sig = {
        "oracle_root_of_unity": [i64, i64, c_int, _D],
        "oracle_dft": [_D, i64, c_int, _D],
        "oracle_dft_bins": [_D, i64, c_int, _I64, i64, _D],
        "oracle_fft": [_D, i64, c_int, _D],
        "oracle_ifft": [_D, i64, _D],
        "oracle_idft": [_D, i64, _D],
        "oracle_fft_batch": [_D, i64, i64, c_int, _D],
        "oracle_fft2d": [_D, i64, i64, c_int, _D],
        "oracle_radix2_pass": [_D, i64, i64, _D],
        "oracle_bit_reverse": [_D, i64, _D],
        "oracle_bit_reverse_index": [i64, i64, _I64],
        "oracle_stockham_stage": [_D, i64, c_int, _D],
        "oracle_polymul_schoolbook_at": [_I64, i64, _I64, i64, _I64, i64, _I64],
        "oracle_polymul_fft": [_I64, i64, _I64, i64, _I64],
        "oracle_poly_eval_mod": [_I64, i64, ctypes.c_uint64, _U64],
        "oracle_convolve": [_D, i64, _D, i64, _D],
        "oracle_rfft": [_D, i64, _D],
        "oracle_irfft": [_D, i64, _D],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB_OVERRIDE: a library built from a deliberately mutated
            # copy of fft_oracle.c, used by the pin-strength tests to show that
            # the pins catch planted mistakes.
            override = os.environ.get("ORACLE_LIB_OVERRIDE")
            if override:
                _lib = bind(ctypes.CDLL(override))
            else:
                build()
                _lib = bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _c128(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.complex128))


def _i64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _ip(a: np.ndarray):
    return a.ctypes.data_as(_I64)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed (rc={rc})")


def root_of_unity(m: int, n: int, sign: int = -1) -> complex:
    """omega_N^m with omega_N = e^{sign i 2 pi / N} ("FFT on GPU", Primitive
    Root of Unity); m reduced mod N in integers first."""
    out = np.zeros(2, dtype=np.float64)
    _check(_load().oracle_root_of_unity(int(m), int(n), int(sign), _dp(out)), "root")
    return complex(out[0], out[1])


def dft(x, direction: int = -1) -> np.ndarray:
    """Direct O(N^2) DFT of a 1D vector (any N >= 1).  direction -1: forward,
    unscaled; +1: inverse with 1/N ("FFT on GPU", DFT definition and the
    inverse formula)."""
    x = _c128(x)
    out = np.empty_like(x)
    if direction < 0:
        _check(_load().oracle_dft(_dp(x), x.size, -1, _dp(out)), "dft")
    else:
        _check(_load().oracle_idft(_dp(x), x.size, _dp(out)), "idft")
    return out


def dft_bins(x, ks, direction: int = -1) -> np.ndarray:
    """Selected bins X_k of the direct DFT, O(N) each (unscaled, either sign)."""
    x = _c128(x)
    ks = _i64(ks)
    out = np.empty(ks.size, dtype=np.complex128)
    _check(_load().oracle_dft_bins(_dp(x), x.size, -1 if direction < 0 else 1, _ip(ks),
                                   ks.size, _dp(out)), "dft_bins")
    return out


def fft(x, direction: int = -1) -> np.ndarray:
    """Recursive even/odd Cooley-Tukey of a 1D power-of-two vector, or of
    every row of a 2D array (batch-contiguous).  direction -1: forward;
    +1: inverse with 1/N."""
    x = _c128(x)
    if x.ndim == 1:
        x2 = x.reshape(1, -1)
    else:
        x2 = x.reshape(-1, x.shape[-1])
    out = np.empty_like(x2)
    _check(_load().oracle_fft_batch(_dp(x2), x2.shape[1], x2.shape[0], -1 if direction < 0 else 1,
                                    _dp(out)), "fft")
    return out.reshape(x.shape)


def ifft(X) -> np.ndarray:
    """Inverse of ``fft``: conjugate root and the factor 1/N."""
    return fft(X, direction=+1)


def fft2d(x, direction: int = -1) -> np.ndarray:
    """Separable 2D transform of one image [h][w] or a batch [b][h][w]:
    rows (contiguous axis) first, then columns.  Inverse scales by 1/(h*w)."""
    x = _c128(x)
    squeeze = x.ndim == 2
    x3 = x.reshape(1, *x.shape) if squeeze else x
    out = np.empty_like(x3)
    lib = _load()
    for b in range(x3.shape[0]):
        src = np.ascontiguousarray(x3[b])
        dst = np.empty_like(src)
        _check(lib.oracle_fft2d(_dp(src), src.shape[0], src.shape[1], -1 if direction < 0 else 1,
                                _dp(dst)), "fft2d")
        out[b] = dst
    return out[0] if squeeze else out


def radix2_pass(x, half: int) -> np.ndarray:
    """One gather-shaped radix-2 butterfly pass at half-block size ``half``."""
    x = _c128(x)
    out = np.empty_like(x)
    _check(_load().oracle_radix2_pass(_dp(x), x.size, int(half), _dp(out)), "radix2_pass")
    return out


def bit_reverse(x) -> np.ndarray:
    """y[i] = x[rev(i)]."""
    x = _c128(x)
    out = np.empty_like(x)
    _check(_load().oracle_bit_reverse(_dp(x), x.size, _dp(out)), "bit_reverse")
    return out


def bit_reverse_index(i: int, n: int) -> int:
    out = ctypes.c_int64(0)
    _check(_load().oracle_bit_reverse_index(int(i), int(n), ctypes.byref(out)), "bitrev index")
    return int(out.value)


def stockham_stage(x, s: int) -> np.ndarray:
    """One forward Stockham stage s (natural order in and out)."""
    x = _c128(x)
    out = np.empty_like(x)
    _check(_load().oracle_stockham_stage(_dp(x), x.size, int(s), _dp(out)), "stockham_stage")
    return out


def polymul_schoolbook_at(a, b, idx) -> np.ndarray:
    """Exact coefficients c_k = sum_i a_i b_{k-i} at the given indices."""
    a, b, idx = _i64(a), _i64(b), _i64(idx)
    out = np.empty(idx.size, dtype=np.int64)
    _check(_load().oracle_polymul_schoolbook_at(_ip(a), a.size, _ip(b), b.size, _ip(idx),
                                                idx.size, _ip(out)), "schoolbook")
    return out


def polymul_schoolbook(a, b) -> np.ndarray:
    a, b = _i64(a), _i64(b)
    return polymul_schoolbook_at(a, b, np.arange(a.size + b.size - 1, dtype=np.int64))


def polymul_fft(a, b) -> np.ndarray:
    """fp64 pipeline: pad to a power of two, transform both, multiply
    pointwise, inverse transform, round.  Returns na+nb-1 coefficients."""
    a, b = _i64(a), _i64(b)
    out = np.empty(a.size + b.size - 1, dtype=np.int64)
    _check(_load().oracle_polymul_fft(_ip(a), a.size, _ip(b), b.size, _ip(out)), "polymul_fft")
    return out


MOD_P = (1 << 61) - 1


def poly_eval_mod(a, t: int) -> int:
    """A(t) mod (2^61 - 1) by Horner's rule."""
    a = _i64(a)
    out = ctypes.c_uint64(0)
    _check(_load().oracle_poly_eval_mod(_ip(a), a.size, ctypes.c_uint64(int(t) % MOD_P),
                                        ctypes.byref(out)), "poly_eval_mod")
    return int(out.value)


def convolve(x, h) -> np.ndarray:
    """Linear convolution y_k = sum_i x_i h_{k-i} of 1D sequences (complex
    or real; returned complex128), or of each row of a 2D x with a 1D h, or
    row-wise with a 2D h of the same number of rows."""
    x = _c128(x)
    h = _c128(h)
    lib = _load()
    if x.ndim == 1 and h.ndim == 1:
        out = np.empty(x.size + h.size - 1, dtype=np.complex128)
        _check(lib.oracle_convolve(_dp(x), x.size, _dp(h), h.size, _dp(out)), "convolve")
        return out
    x2 = x.reshape(-1, x.shape[-1])
    rows = []
    for r in range(x2.shape[0]):
        hr = h if h.ndim == 1 else np.ascontiguousarray(h.reshape(-1, h.shape[-1])[r])
        rows.append(convolve(np.ascontiguousarray(x2[r]), hr))
    return np.stack(rows)


def _transform_rows(x2: np.ndarray, direction: int) -> np.ndarray:
    """1D transform of every row: the recursive CT for power-of-two lengths,
    the direct DFT for the others."""
    n = x2.shape[-1]
    if n & (n - 1) == 0:
        return fft(x2, direction)
    return np.stack([dft(np.ascontiguousarray(r), direction) for r in x2.reshape(-1, n)]
                    ).reshape(x2.shape)


def fftn(x, ndim: int, direction: int = -1) -> np.ndarray:
    """The 1D transform along each of the last `ndim` axes in turn, the
    contiguous axis first (separable transform): recursive CT for
    power-of-two sides, direct DFT for the others; the inverse scales by
    1/(product of the sides).  numpy only moves axes; the arithmetic is the
    oracle's."""
    y = _c128(x)
    for k in range(1, ndim + 1):
        axis = y.ndim - k
        moved = np.ascontiguousarray(np.moveaxis(y, axis, -1))
        y = np.moveaxis(_transform_rows(moved, direction), -1, axis)
    return np.ascontiguousarray(y)


def rfft(x) -> np.ndarray:
    """Half spectrum X_k, k = 0 .. n//2, of each real row (last axis) of x:
    the first n//2 + 1 bins of its DFT (forward, unscaled)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    n = x.shape[-1]
    x2 = x.reshape(-1, n)
    out = np.empty((x2.shape[0], n // 2 + 1), dtype=np.complex128)
    lib = _load()
    for r in range(x2.shape[0]):
        row = np.ascontiguousarray(x2[r])
        res = np.empty(n // 2 + 1, dtype=np.complex128)
        _check(lib.oracle_rfft(_dp(row), n, _dp(res)), "rfft")
        out[r] = res
    return out.reshape(x.shape[:-1] + (n // 2 + 1,))


def irfft(X, n: int) -> np.ndarray:
    """Real rows of length n from half spectra X[..., n//2 + 1]: the inverse
    transform (1/n) of the Hermitian extension, real part."""
    X = _c128(X)
    if X.shape[-1] != n // 2 + 1:
        raise ValueError("half spectrum must have n//2 + 1 bins")
    X2 = X.reshape(-1, X.shape[-1])
    out = np.empty((X2.shape[0], n), dtype=np.float64)
    lib = _load()
    for r in range(X2.shape[0]):
        row = np.ascontiguousarray(X2[r])
        res = np.empty(n, dtype=np.float64)
        _check(lib.oracle_irfft(_dp(row), n, _dp(res)), "irfft")
        out[r] = res
    return out.reshape(X.shape[:-1] + (n,))
