"""Pins for the fp64 CPU oracle (CPU only).

Every oracle function is checked against something other than itself: values
the pages print, closed forms, the root-of-unity identities, invariants of
the DFT, numpy's own FFT (an independent library the oracle does not call),
and exact big-integer arithmetic for the polynomial product.  The cases are
chosen so that a dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

POW2 = [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024]


def rel_l2(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


# --- DFT definition ("FFT on GPU", Discrete Fourier Transform) -------------

@pytest.mark.parametrize("n", POW2)
def test_delta_gives_all_ones(n):
    x = np.zeros(n, complex)
    x[0] = 1
    assert np.array_equal(oracle.dft(x), np.ones(n))
    assert np.array_equal(oracle.fft(x), np.ones(n))


@pytest.mark.parametrize("n", [2, 8, 64, 1024])
def test_constant_gives_n_at_bin0(n):
    c = 0.75 - 0.25j
    x = np.full(n, c)
    for X in (oracle.dft(x), oracle.fft(x)):
        assert abs(X[0] - n * c) < 1e-12 * n
        assert np.max(np.abs(X[1:])) < 1e-12 * n


@pytest.mark.parametrize("n,f", [(8, 1), (8, 3), (64, 5), (1024, 317), (1024, 1023)])
def test_single_tone_lands_in_one_bin(n, f):
    # x_n = e^{+i 2 pi f n / N}; forward transform is N at bin f, 0 elsewhere.
    k = (f * np.arange(n)) % n
    x = np.exp(2j * np.pi * k / n)
    expect = np.zeros(n, complex)
    expect[f] = n
    for X in (oracle.dft(x), oracle.fft(x)):
        assert np.max(np.abs(X - expect)) < 1e-11 * n


def test_closed_forms_n2_n4():
    # Hand-derived from the definition with omega_4 = -i.
    a = workloads.uniform_complex(2, 11, np.complex128)
    X = oracle.fft(a)
    assert np.allclose(X, [a[0] + a[1], a[0] - a[1]], atol=1e-15)
    assert np.allclose(oracle.dft(a), X, atol=1e-15)
    a = workloads.uniform_complex(4, 12, np.complex128)
    expect = [a[0] + a[1] + a[2] + a[3],
              a[0] - 1j * a[1] - a[2] + 1j * a[3],
              a[0] - a[1] + a[2] - a[3],
              a[0] + 1j * a[1] - a[2] - 1j * a[3]]
    for X in (oracle.dft(a), oracle.fft(a)):
        assert np.allclose(X, expect, atol=1e-15)


@pytest.mark.parametrize("n", [2, 16, 128, 1024, 4096])
def test_direct_dft_and_cooley_tukey_agree(n):
    x = workloads.normal_complex(n, 100 + n, np.complex128)
    d = oracle.dft(x)
    c = oracle.fft(x)
    assert rel_l2(c, d) < 1e-13


@pytest.mark.parametrize("n", [1, 2, 8, 256, 2048, 1 << 15])
def test_matches_numpy_fft(n):
    # numpy.fft is an independent implementation the oracle never calls.
    x = workloads.normal_complex(n, 200 + n, np.complex128)
    assert rel_l2(oracle.fft(x), np.fft.fft(x)) < 1e-14
    assert rel_l2(oracle.ifft(x), np.fft.ifft(x)) < 1e-14
    if n <= 2048:
        assert rel_l2(oracle.dft(x), np.fft.fft(x)) < 1e-14
        assert rel_l2(oracle.dft(x, +1), np.fft.ifft(x)) < 1e-14


def test_dft_bins_match_full_transform():
    n = 1 << 14
    x = workloads.normal_complex(n, 7, np.complex128)
    ks = workloads.sample_indices(40, n, 8)
    ref = np.fft.fft(x)[ks]
    assert rel_l2(oracle.dft_bins(x, ks), ref) < 1e-13
    refi = np.fft.ifft(x)[ks] * n
    assert rel_l2(oracle.dft_bins(x, ks, +1), refi) < 1e-13


# --- invariants --------------------------------------------------------------

@pytest.mark.parametrize("n", [4, 256, 4096])
def test_parseval(n):
    x = workloads.normal_complex(n, 300 + n, np.complex128)
    X = oracle.fft(x)
    assert abs(np.sum(np.abs(x) ** 2) - np.sum(np.abs(X) ** 2) / n) < 1e-11 * n


@pytest.mark.parametrize("n", [1, 2, 32, 4096])
def test_round_trip(n):
    x = workloads.normal_complex(n, 400 + n, np.complex128)
    assert rel_l2(oracle.ifft(oracle.fft(x)), x) < 1e-14
    if n <= 1024:
        assert rel_l2(oracle.dft(oracle.dft(x), +1), x) < 1e-14


def test_linearity():
    n = 512
    x = workloads.normal_complex(n, 1, np.complex128)
    y = workloads.normal_complex(n, 2, np.complex128)
    a, b = 0.3 - 1.1j, -2.0 + 0.5j
    lhs = oracle.fft(a * x + b * y)
    rhs = a * oracle.fft(x) + b * oracle.fft(y)
    assert rel_l2(lhs, rhs) < 1e-14


@pytest.mark.parametrize("n", [8, 1024])
def test_hermitian_symmetry_of_real_input(n):
    x = workloads.normal_complex(n, 5, np.complex128).real.astype(complex)
    X = oracle.fft(x)
    k = np.arange(1, n)
    assert np.max(np.abs(X[n - k] - np.conj(X[k]))) < 1e-12 * n
    assert abs(X[0].imag) < 1e-12 * n


# --- roots of unity ("FFT on GPU", Primitive Root of Unity) -----------------

@pytest.mark.parametrize("n", [2, 8, 64, 4096, 1 << 26])
def test_root_of_unity_identities(n):
    ks = sorted(set([0, 1, 2, 3, n // 4, n // 2 - 1, n - 1] + list(range(0, n, max(1, n // 17)))))
    for k in ks:
        w = oracle.root_of_unity(k, n)
        assert abs(abs(w) - 1) < 1e-15
        assert abs(oracle.root_of_unity(k + n, n) - w) < 1e-15          # periodicity
        assert abs(oracle.root_of_unity(k + n // 2, n) + w) < 1e-15     # symmetry
        if n >= 2:
            assert abs(oracle.root_of_unity(2 * k, n) - oracle.root_of_unity(k, n // 2)) < 1e-15
    assert abs(oracle.root_of_unity(1, 4) - (-1j)) < 1e-16              # omega_4 = -i
    assert abs(oracle.root_of_unity(1, 4, +1) - 1j) < 1e-16


# --- the single butterfly pass (gpu.rocks, task 2) ---------------------------

def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_p1_pairing_at_half2(golden_dir):
    g = _golden(golden_dir, "p1_pairs.json")
    n = g["n"]
    # A unit impulse at position p only reaches the two cells of p's pair.
    for lower in g["half2_lower_j0"]:
        upper = lower + 2
        assert upper in g["half2_upper_j1"]
        for p in (lower, upper):
            x = np.zeros(n, complex)
            x[p] = 1
            y = oracle.radix2_pass(x, 2)
            assert set(np.nonzero(np.abs(y) > 1e-14)[0]) == {lower, upper}
    # The lower member receives a + w b, the upper a - w b: impulse at the
    # upper index r = 1 gives w = e^{-i pi/2} = -i at the lower cell.
    x = np.zeros(n, complex)
    x[3] = 1
    y = oracle.radix2_pass(x, 2)
    assert abs(y[1] - (-1j)) < 1e-15 and abs(y[3] - 1j) < 1e-15


def test_p1_half1_is_pure_add_sub(golden_dir):
    g = _golden(golden_dir, "p1_pairs.json")
    assert g["half1_twiddle"] == [1.0, 0.0]
    x = workloads.p1_spectrum()
    y = oracle.radix2_pass(x, 1)
    expect = np.empty(8, complex)
    expect[0::2] = x[0::2] + x[1::2]
    expect[1::2] = x[0::2] - x[1::2]
    assert np.array_equal(y, expect)


@pytest.mark.parametrize("half", [1, 2, 4])
def test_p1_single_pass_closed_form(half):
    # Each output is written out from the recipe's two inputs and twiddle.
    x = workloads.p1_spectrum()
    y = oracle.radix2_pass(x, half)
    for i in range(8):
        blk = 2 * half
        lo = (i // blk) * blk + (i % half)
        r = i % half
        w = np.exp(-1j * np.pi * r / half)
        want = x[lo] + w * x[lo + half] if (i % blk) < half else x[lo] - w * x[lo + half]
        assert abs(y[i] - want) < 1e-15


def test_bit_reverse_golden(golden_dir):
    g = _golden(golden_dir, "bitrev8.json")
    assert [oracle.bit_reverse_index(i, 8) for i in range(8)] == g["order"]
    assert [format(v, "03b") for v in g["order"]] == g["bits"]
    x = np.arange(8) + 0j
    assert np.array_equal(oracle.bit_reverse(x).real.astype(int), g["order"])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bitrev_then_passes_is_dft8(seed):
    x = workloads.p1_spectrum(seed)
    y = oracle.bit_reverse(x)
    for half in (1, 2, 4):
        y = oracle.radix2_pass(y, half)
    assert rel_l2(y, np.fft.fft(x)) < 1e-15
    # Ramp input too (x_n = n).
    r = np.arange(8) + 0j
    y = oracle.bit_reverse(r)
    for half in (1, 2, 4):
        y = oracle.radix2_pass(y, half)
    assert rel_l2(y, np.fft.fft(r)) < 1e-15


def test_passes_on_natural_order_are_not_the_dft():
    x = workloads.p1_spectrum()
    y = x.copy()
    for half in (1, 2, 4):
        y = oracle.radix2_pass(y, half)
    assert rel_l2(y, np.fft.fft(x)) > 0.1
    assert rel_l2(oracle.bit_reverse(y), np.fft.fft(x)) > 0.1


# --- Stockham stages (salivity GLSL page) -----------------------------------

@pytest.mark.parametrize("n", [2, 4, 8, 64, 1024])
def test_stockham_stages_compose_to_dft(n):
    x = workloads.normal_complex(n, 500 + n, np.complex128)
    y = x
    for s in range(n.bit_length() - 1):
        y = oracle.stockham_stage(y, s)
    assert rel_l2(y, np.fft.fft(x)) < 1e-14


# --- 2D ---------------------------------------------------------------------

@pytest.mark.parametrize("h,w", [(1, 1), (2, 8), (16, 16), (64, 32)])
def test_fft2d_matches_numpy(h, w):
    x = workloads.normal_complex((3, h, w), 600 + h * w, np.complex128)
    X = oracle.fft2d(x)
    assert rel_l2(X, np.fft.fft2(x)) < 1e-14
    assert rel_l2(oracle.fft2d(X, +1), x) < 1e-14
    d = np.zeros((h, w), complex)
    d[0, 0] = 1
    assert np.array_equal(oracle.fft2d(d), np.ones((h, w)))


# --- polynomial multiplication ("FFT on GPU", polynomial section) ----------

def _kronecker(a, b, base_digits=6):
    # Independent exact product: evaluate at x = 10^d with Python big
    # integers and read the base-10^d digits (valid for 0 <= c_k < 10^d).
    base = 10 ** base_digits
    A = sum(int(v) * base ** i for i, v in enumerate(a))
    B = sum(int(v) * base ** i for i, v in enumerate(b))
    C = A * B
    out = []
    for _ in range(len(a) + len(b) - 1):
        C, r = divmod(C, base)
        out.append(r)
    return np.array(out, dtype=np.int64)


def test_polymul_tiny_exhaustive():
    for na in range(1, 5):
        for nb in range(1, 4):
            for a_val in range(0, 10, 3):
                for b_val in range(0, 10, 4):
                    a = (np.arange(na) * 7 + a_val) % 10
                    b = (np.arange(nb) * 3 + b_val) % 10
                    ref = _kronecker(a, b)
                    assert np.array_equal(oracle.polymul_schoolbook(a, b), ref)
                    assert np.array_equal(oracle.polymul_fft(a, b), ref)


@pytest.mark.parametrize("n", [1, 2, 3, 16, 100, 1000])
def test_polymul_random_against_big_integers(n):
    a, b = workloads.poly_coeffs(n, 700 + n)
    ref = _kronecker(a, b)
    assert np.array_equal(oracle.polymul_schoolbook(a, b), ref)
    assert np.array_equal(oracle.polymul_fft(a, b), ref)


def test_polymul_eval_at_plus_minus_one():
    a, b = workloads.poly_coeffs(257, 9)
    c = oracle.polymul_fft(a, b)
    sgn = lambda m: (-1) ** np.arange(m)
    assert c.sum() == a.sum() * b.sum()
    assert (c * sgn(c.size)).sum() == (a * sgn(a.size)).sum() * (b * sgn(b.size)).sum()


def test_polymul_mixed_sign_coefficients():
    g = workloads.generator(31)
    a = g.integers(-1000, 1000, size=50)
    b = g.integers(-1000, 1000, size=70)
    want = np.convolve(a.astype(object), b.astype(object)).astype(np.int64)
    assert np.array_equal(oracle.polymul_schoolbook(a, b), want)
    assert np.array_equal(oracle.polymul_fft(a, b), want)


def test_poly_eval_mod_matches_big_integers():
    P = oracle.MOD_P
    g = workloads.generator(41)
    a = g.integers(-(1 << 62), 1 << 62, size=33)
    for t in (0, 1, 2, 12345678901234567, P - 1):
        want = sum(int(v) * pow(t, i, P) for i, v in enumerate(a)) % P
        assert oracle.poly_eval_mod(a, t) == want


def test_polymul_modular_identity_at_size():
    a, b = workloads.poly_coeffs(4096, 51)
    c = oracle.polymul_fft(a, b)
    for t in workloads.sample_indices(4, oracle.MOD_P, 52):
        t = int(t)
        lhs = oracle.poly_eval_mod(c, t)
        rhs = oracle.poly_eval_mod(a, t) * oracle.poly_eval_mod(b, t) % oracle.MOD_P
        assert lhs == rhs
    idx = workloads.sample_indices(64, c.size, 53)
    assert np.array_equal(oracle.polymul_schoolbook_at(a, b, idx), c[idx])


# --- seeded inputs ------------------------------------------------------------

def test_workloads_are_deterministic():
    assert np.array_equal(workloads.normal_complex((4, 8), 3), workloads.normal_complex((4, 8), 3))
    assert not np.array_equal(workloads.normal_complex(8, 3), workloads.normal_complex(8, 4))
    a1, b1 = workloads.poly_coeffs(100, 5)
    a2, b2 = workloads.poly_coeffs(100, 5)
    assert np.array_equal(a1, a2) and np.array_equal(b1, b2)
    assert a1.min() >= 0 and a1.max() <= 9


def test_tones_signal_spectrum():
    # Small instance of the tone workload: 16 tones of unit amplitude land
    # in their own bins with magnitude N, noise spreads ~sigma*sqrt(N).
    n = 1 << 12
    bins, phases, _ = workloads.tone_params(n, 77)
    x = workloads.tones_plus_noise(n, 77, dtype=np.complex128)
    X = np.abs(np.fft.fft(x))
    assert np.all(np.abs(X[bins] - n) < 8 * 0.1 * np.sqrt(2 * n))
    mask = np.ones(n, bool)
    mask[bins] = False
    assert X[mask].max() < 8 * 0.1 * np.sqrt(2 * n)


# --- linear convolution of signals ------------------------------------------

@pytest.mark.parametrize("nx,nh", [(1, 1), (5, 3), (64, 17), (300, 1000)])
def test_convolve_matches_numpy(nx, nh):
    x = workloads.normal_complex(nx, nx, np.complex128)
    h = workloads.normal_complex(nh, nh + 1, np.complex128)
    y = oracle.convolve(x, h)
    assert y.size == nx + nh - 1
    assert rel_l2(y, np.convolve(x, h)) < 1e-14


def test_convolve_delta_shift_commute_linear():
    x = workloads.uniform_complex(50, 3, np.complex128)
    h = workloads.uniform_complex(20, 4, np.complex128)
    d = np.zeros(7, complex)
    d[0] = 1
    assert np.array_equal(oracle.convolve(x, d)[:50], x)               # delta is the identity
    d = np.zeros(7, complex)
    d[4] = 1
    y = oracle.convolve(x, d)
    assert np.array_equal(y[4:54], x) and np.all(y[:4] == 0)          # shifted delta shifts
    assert rel_l2(oracle.convolve(x, h), oracle.convolve(h, x)) < 1e-15  # commutes
    g = workloads.uniform_complex(50, 5, np.complex128)
    lhs = oracle.convolve(2 * x - 1j * g, h)
    assert rel_l2(lhs, 2 * oracle.convolve(x, h) - 1j * oracle.convolve(g, h)) < 1e-14


def test_convolve_of_integers_is_the_polynomial_product():
    a, b = workloads.poly_coeffs(40, 6)
    y = oracle.convolve(a.astype(float), b.astype(float))
    assert np.array_equal(np.rint(y.real).astype(np.int64), oracle.polymul_schoolbook(a, b))
    assert np.max(np.abs(y.imag)) == 0


def test_convolve_rows():
    x = workloads.normal_complex((3, 40), 7, np.complex128)
    h = workloads.normal_complex((3, 9), 8, np.complex128)
    y = oracle.convolve(x, h)
    for r in range(3):
        assert rel_l2(y[r], np.convolve(x[r], h[r])) < 1e-14
    y1 = oracle.convolve(x, h[0])
    assert rel_l2(y1[2], np.convolve(x[2], h[0])) < 1e-14


@pytest.mark.parametrize("shape", [(2, 8), (16, 4), (4, 8, 16), (2, 1, 32), (8, 8, 8),
                                   (3, 5), (6, 10), (12, 7, 9), (1, 100), (5, 1, 3)])
def test_fftn_matches_numpy(shape):
    x = workloads.normal_complex((2,) + shape, 900 + len(shape), np.complex128)
    nd = len(shape)
    X = oracle.fftn(x, nd)
    assert rel_l2(X, np.fft.fftn(x, axes=tuple(range(-nd, 0)))) < 1e-14
    assert rel_l2(oracle.fftn(X, nd, +1), x) < 1e-14
    d = np.zeros(shape, complex)
    d[(0,) * nd] = 1
    assert np.array_equal(oracle.fftn(d, nd), np.ones(shape))
    if nd == 2 and all(v & (v - 1) == 0 for v in shape):
        assert rel_l2(X, oracle.fft2d(x)) < 1e-15


# --- lengths that are not powers of two (direct DFT) ------------------------

@pytest.mark.parametrize("n", [3, 5, 6, 12, 97, 1000])
def test_direct_dft_any_length_matches_numpy(n):
    x = workloads.normal_complex(n, 1100 + n, np.complex128)
    assert rel_l2(oracle.dft(x), np.fft.fft(x)) < 1e-13
    assert rel_l2(oracle.dft(x, +1), np.fft.ifft(x)) < 1e-13


def test_direct_dft_closed_form_n3():
    # omega_3 = e^{-2 pi i / 3} = -1/2 - i sqrt(3)/2; X_k = sum_n x_n omega^{kn}.
    a = workloads.uniform_complex(3, 13, np.complex128)
    w = -0.5 - 0.5j * np.sqrt(3.0)
    expect = [a[0] + a[1] + a[2], a[0] + w * a[1] + w * w * a[2], a[0] + w * w * a[1] + w * a[2]]
    assert np.allclose(oracle.dft(a), expect, atol=1e-14)


# --- transforms of real sequences (half spectrum) ---------------------------
# Derived from the DFT definition ("FFT on GPU", Discrete Fourier Transform)
# for real samples, which the page's polynomial section uses (real
# coefficients): X_{N-k} = conj(X_k).

RLEN = [1, 2, 3, 4, 7, 8, 64, 100, 1024]


@pytest.mark.parametrize("n", RLEN)
def test_rfft_matches_numpy(n):
    x = workloads.generator(1200 + n).standard_normal(size=(3, n))
    X = oracle.rfft(x)
    assert X.shape == (3, n // 2 + 1)
    assert rel_l2(X, np.fft.rfft(x, axis=-1)) < 1e-13


@pytest.mark.parametrize("n", RLEN)
def test_irfft_matches_numpy(n):
    g = workloads.generator(1300 + n)
    X = g.standard_normal(size=(3, n // 2 + 1)) + 1j * g.standard_normal(size=(3, n // 2 + 1))
    x = oracle.irfft(X, n)
    assert x.shape == (3, n) and x.dtype == np.float64
    assert rel_l2(x, np.fft.irfft(X, n, axis=-1)) < 1e-13


def test_rfft_closed_forms():
    a = np.array([0.75, -2.5])
    assert np.allclose(oracle.rfft(a), [a[0] + a[1], a[0] - a[1]], atol=0)
    x = np.array([1.0, 2.0, -3.0, 0.5])
    # X_1 = x0 - i x1 - x2 + i x3, X_2 = x0 - x1 + x2 - x3.
    expect = [x.sum(), x[0] - x[2] - 1j * (x[1] - x[3]), x[0] - x[1] + x[2] - x[3]]
    assert np.allclose(oracle.rfft(x), expect, atol=1e-15)
    d = np.zeros(16)
    d[0] = 1.0
    assert np.array_equal(oracle.rfft(d), np.ones(9))
    c = np.full(16, -1.25)
    expect = np.zeros(9, complex)
    expect[0] = 16 * -1.25
    assert np.allclose(oracle.rfft(c), expect, atol=1e-14)


@pytest.mark.parametrize("n,f", [(64, 5), (1024, 300), (100, 7)])
def test_rfft_of_cosine_is_one_bin(n, f):
    # cos(2 pi f k / N) = (w^{-fk} + w^{fk}) / 2: N/2 at bin f, nothing else.
    k = np.arange(n)
    x = np.cos(2 * np.pi * ((f * k) % n) / n)
    expect = np.zeros(n // 2 + 1, complex)
    expect[f] = n / 2
    assert np.abs(oracle.rfft(x) - expect).max() < 1e-11


@pytest.mark.parametrize("n", [2, 8, 1024, 100, 63])
def test_real_round_trip_and_parseval(n):
    x = workloads.generator(1400 + n).standard_normal(size=n)
    X = oracle.rfft(x)
    assert rel_l2(oracle.irfft(X, n), x) < 1e-14
    # Parseval with the mirrored bins counted twice.
    w = np.full(X.size, 2.0)
    w[0] = 1.0
    if n % 2 == 0:
        w[-1] = 1.0
    assert abs(np.sum(w * np.abs(X) ** 2) / n - np.sum(x ** 2)) < 1e-11 * np.sum(x ** 2)


@pytest.mark.parametrize("n", [8, 9, 1024])
def test_irfft_drops_imaginary_dc_and_nyquist(n):
    g = workloads.generator(1500 + n)
    X = g.standard_normal(size=n // 2 + 1) + 1j * g.standard_normal(size=n // 2 + 1)
    clean = X.copy()
    clean[0] = clean[0].real
    if n % 2 == 0:
        clean[-1] = clean[-1].real
    assert rel_l2(oracle.irfft(X, n), oracle.irfft(clean, n)) < 1e-15
    if n % 2 == 1:
        # Odd n has no Nyquist bin: the last bin's imaginary part counts.
        bumped = clean.copy()
        bumped[-1] += 1j
        assert rel_l2(oracle.irfft(bumped, n), oracle.irfft(clean, n)) > 1e-3
