"""Seeded synthetic inputs for the FFT, 2D FFT and polynomial-multiplication
workloads.

This module is the one piece shared by the tests, the smoke check and the
bench on both sides of every comparison (CUDA path and oracle).  It holds
none of the transform arithmetic: only random draws (numpy
``Generator(PCG64(seed))``) and the synthesis of the test signals.  The same
bytes go to the GPU and to the oracle.

Workloads (sizes and distributions):

* ``c1``: one 1024-point transform, fp32, re and im i.i.d. uniform[-1, 1);
  plus the 8-point butterfly-pass unit check (``p1_spectrum``).
* ``c2``: 16384 transforms of 4096 points (512 MiB fp32 complex), re and im
  i.i.d. standard normal; forward, then inverse with 1/N.
* ``c3``: one 2^26-point transform (512 MiB fp32 complex): 16 unit-amplitude
  tones at distinct integer bins with uniform random phase, plus complex
  Gaussian noise with variance 0.01 on each of re and im (sigma = 0.1).
* ``c4``: 8 images of 2048 x 2048 fp32 complex, re and im i.i.d. standard
  normal; forward 2D, then the inverse round trip.
* ``c5``: 64 pairs of polynomials with 2^20 integer coefficients each,
  uniform on {0, ..., 9}; products have 2^21 - 1 coefficients.
* ``conv1``: 32768 real fp32 signals of 3072 samples, i.i.d. standard
  normal, convolved with one shared 1025-tap real filter (standard normal);
  outputs have 4096 samples (transform length 4096).
* ``any1``: 16384 transforms of 3000 = 2^3 3 5^3 points, fp32, re and im
  i.i.d. standard normal; forward then inverse.
* ``any2``: the same with the prime length 3001.
* ``any3``: 1024 transforms of 100000 = 2^5 5^5 points, fp32, N(0, 1).
* ``nd1``: 4 volumes of 128 x 256 x 256 fp32 complex (256 MiB), standard
  normal; 3D forward then inverse.
* ``real1``: 32768 real fp32 rows of 8192 samples (1 GiB), standard normal;
  half spectrum (R2C) then back (C2R).
* ``rows512``: 131072 transforms of 512 points (512 MiB fp32 complex), re and
  im i.i.d. standard normal; forward then inverse (the shape on which the
  shared-memory and warp-shuffle exchanges of the on-chip engine are
  compared).
"""
from __future__ import annotations

import numpy as np

CONFIGS = {
    "c1": dict(kind="fft1d", n=1024, batch=1, dtype="f32", seed=1),
    "c2": dict(kind="fft1d", n=4096, batch=16384, dtype="f32", seed=2),
    "c3": dict(kind="fft1d", n=1 << 26, batch=1, dtype="f32", seed=3),
    "c4": dict(kind="fft2d", n=2048, batch=8, dtype="f32", seed=4),
    "c5": dict(kind="polymul", n=1 << 20, batch=64, dtype="f64", seed=5),
    "conv1": dict(kind="conv", n=3072, nh=1025, batch=32768, dtype="f32", seed=6),
    "any1": dict(kind="fft1d", n=3000, batch=16384, dtype="f32", seed=7),
    "any2": dict(kind="fft1d", n=3001, batch=16384, dtype="f32", seed=10),
    "any3": dict(kind="fft1d", n=100000, batch=1024, dtype="f32", seed=11),
    "nd1": dict(kind="fftnd", n=256, shape=(128, 256, 256), batch=4, dtype="f32", seed=8),
    "real1": dict(kind="real", n=8192, batch=32768, dtype="f32", seed=9),
    "rows512": dict(kind="fft1d", n=512, batch=131072, dtype="f32", seed=12),
}


def generator(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def _complex(re: np.ndarray, im: np.ndarray, dtype) -> np.ndarray:
    out = np.empty(re.shape, dtype=dtype)
    out.real = re
    out.imag = im
    return out


def uniform_complex(shape, seed: int, dtype=np.complex64) -> np.ndarray:
    """re, im i.i.d. uniform on [-1, 1)."""
    g = generator(seed)
    re = g.uniform(-1.0, 1.0, size=shape)
    im = g.uniform(-1.0, 1.0, size=shape)
    return _complex(re, im, dtype)


def normal_complex(shape, seed: int, dtype=np.complex64) -> np.ndarray:
    """re, im i.i.d. standard normal.  Drawn directly in float32 when the
    target is complex64 (half the memory and time at 512 MiB sizes)."""
    g = generator(seed)
    if np.dtype(dtype) == np.complex64:
        re = g.standard_normal(size=shape, dtype=np.float32)
        im = g.standard_normal(size=shape, dtype=np.float32)
    else:
        re = g.standard_normal(size=shape)
        im = g.standard_normal(size=shape)
    return _complex(re, im, dtype)


def normal_real(shape, seed: int, dtype=np.float32) -> np.ndarray:
    """i.i.d. standard normal real samples (drawn in the target precision)."""
    g = generator(seed)
    if np.dtype(dtype) == np.float32:
        return g.standard_normal(size=shape, dtype=np.float32)
    return g.standard_normal(size=shape).astype(dtype)


def tone_params(n: int, seed: int, ntones: int = 16):
    """The tones' integer bins (distinct, uniform in [0, n)) and phases
    (uniform in [0, 1) turns)."""
    g = generator(seed)
    ntones = min(ntones, n)
    bins = np.sort(g.choice(n, size=ntones, replace=False)).astype(np.int64)
    phases = g.uniform(0.0, 1.0, size=ntones)
    return bins, phases, g


def tones_plus_noise(n: int, seed: int, ntones: int = 16, sigma: float = 0.1,
                     dtype=np.complex64) -> np.ndarray:
    """sum_t exp(i 2 pi (f_t n / N + phi_t)) + complex Gaussian noise.

    Synthesised in fp64 as a rank-``ntones`` outer product over a split
    n = hi * n_lo + lo, with every phase index reduced mod N in integers:
    exp(i 2 pi f (hi n_lo + lo) / N) = exp(i 2 pi f hi n_lo / N) exp(i 2 pi f lo / N).
    """
    bins, phases, g = tone_params(n, seed, ntones)
    log_n = int(n).bit_length() - 1
    n_lo = 1 << ((log_n + 1) // 2)
    n_hi = n // n_lo
    hi = np.arange(n_hi, dtype=np.int64)
    lo = np.arange(n_lo, dtype=np.int64)
    a = np.exp(2j * np.pi * (((bins[None, :] * hi[:, None] * n_lo) % n) / n))
    b = np.exp(2j * np.pi * (((bins[:, None] * lo[None, :]) % n) / n + phases[:, None]))
    x = (a @ b).reshape(n)
    noise_re = g.standard_normal(size=n) * sigma
    noise_im = g.standard_normal(size=n) * sigma
    return _complex(x.real + noise_re, x.imag + noise_im, dtype)


def poly_coeffs(shape, seed: int, lo: int = 0, hi: int = 9):
    """Two integer coefficient arrays a, b of the given shape, uniform on
    {lo, ..., hi}."""
    g = generator(seed)
    a = g.integers(lo, hi + 1, size=shape, dtype=np.int64)
    b = g.integers(lo, hi + 1, size=shape, dtype=np.int64)
    return a, b


def sample_indices(count: int, upper: int, seed: int) -> np.ndarray:
    """``count`` indices uniform in [0, upper) (with repetition)."""
    return generator(seed).integers(0, upper, size=count, dtype=np.int64)


def p1_spectrum(seed: int = 0) -> np.ndarray:
    """The 8-point complex vector for the single-pass unit check.  The
    butterfly page takes its ``spectrum`` from an earlier task that it does
    not print; it is read here as a seeded uniform[-1, 1) vector."""
    return uniform_complex(8, seed, dtype=np.complex128)


def config_input(name: str, scale_batch: int | None = None):
    """The input of one workload (host numpy arrays).  ``scale_batch``
    replaces the batch (for bounded samples of the same workload)."""
    c = CONFIGS[name]
    batch = c["batch"] if scale_batch is None else scale_batch
    if name == "c1":
        return uniform_complex((batch, c["n"]), c["seed"])
    if name == "c2":
        return normal_complex((batch, c["n"]), c["seed"])
    if name == "c3":
        return tones_plus_noise(c["n"], c["seed"]).reshape(1, c["n"])
    if name == "c4":
        return normal_complex((batch, c["n"], c["n"]), c["seed"])
    if name == "c5":
        return poly_coeffs((batch, c["n"]), c["seed"])
    if name == "conv1":
        return conv_signals(batch, c["n"], c["nh"], c["seed"])
    if name in ("any1", "any2", "any3", "rows512"):
        return normal_complex((batch, c["n"]), c["seed"])
    if name == "nd1":
        return normal_complex((batch,) + tuple(c["shape"]), c["seed"])
    if name == "real1":
        return normal_real((batch, c["n"]), c["seed"])
    raise KeyError(name)


def conv_signals(batch: int, n: int, nh: int, seed: int):
    """Real fp32 signals [batch, n] and one real fp32 filter [nh], i.i.d.
    standard normal."""
    g = generator(seed)
    x = g.standard_normal(size=(batch, n), dtype=np.float32)
    h = g.standard_normal(size=nh, dtype=np.float32)
    return x, h
