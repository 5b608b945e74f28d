"""Strength of the oracle's pins: plausible mistakes planted in a copy of
fft_oracle.c (a flipped sign, a wrong or shifted index, a dropped term, halves
swapped, a wrong scale, truncation for rounding) must each make the pin suite
(tests/test_oracle.py) fail.  Every mutant is compiled on the CPU and run
through the pins in a subprocess; the unmutated copy must pass."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fft_oracle.c")

# (name, text in fft_oracle.c, replacement)
MUTANTS = [
    ("root of unity: sign of the sine flipped",
     "return cos(ang) + (double)sign * sin(ang) * I;",
     "return cos(ang) - (double)sign * sin(ang) * I;"),
    ("Cooley-Tukey: upper output gets e + o",
     "X[k + h] = e - o;", "X[k + h] = e + o;"),
    ("Cooley-Tukey: twiddle index off by one",
     "cplx o = root_of_unity(k, n, sign) * X[k + h];",
     "cplx o = root_of_unity(k + 1, n, sign) * X[k + h];"),
    ("Cooley-Tukey: odd half computed from the even samples",
     "ct_recursive(x + stride, 2 * stride, h, sign, X + h);",
     "ct_recursive(x, 2 * stride, h, sign, X + h);"),
    ("direct DFT: exponent index shifted",
     "root_of_unity(mulmod(kk, j, n), n, sign)",
     "root_of_unity(mulmod(kk, (j + 1) % n, n), n, sign)"),
    ("direct DFT: first term dropped",
     "    for (int64_t j = 0; j < n; ++j) {\n        cplx term",
     "    for (int64_t j = 1; j < n; ++j) {\n        cplx term"),
    ("inverse: 1/(N+1) instead of 1/N",
     "int rc = oracle_fft(X, n, +1, x);\n    if (rc) return rc;\n    double s = 1.0 / (double)n;",
     "int rc = oracle_fft(X, n, +1, x);\n    if (rc) return rc;\n    double s = 1.0 / (double)(n + 1);"),
    ("2D: rows transformed with the wrong sign",
     "ct_recursive(xc + r * w, 1, w, sign, tmp);",
     "ct_recursive(xc + r * w, 1, w, -sign, tmp);"),
    ("butterfly pass: base not shifted by half",
     "int64_t base = i - j * half;", "int64_t base = i - j;"),
    ("butterfly pass: twiddle conjugated",
     "cplx wb = root_of_unity(r, 2 * half, -1) * b;",
     "cplx wb = root_of_unity(r, 2 * half, +1) * b;"),
    ("bit reversal: wrong bit taken",
     "rev = (rev << 1) | (t & 1);", "rev = (rev << 1) | ((t >> 1) & 1);"),
    ("Stockham stage: twiddle from the half-block position",
     "int64_t r = (xi % span) * (n / span);", "int64_t r = (xi % half) * (n / span);"),
    ("schoolbook: one product counted twice",
     "for (int64_t i = lo; i <= hi; ++i) s += (__int128)a[i] * (__int128)b[k - i];",
     "for (int64_t i = lo; i <= hi; ++i) s += (__int128)a[i] * (__int128)b[k - i];\n        s += (__int128)a[lo] * (__int128)b[k - lo];"),
    ("polymul pipeline: truncation instead of rounding",
     "c[k] = llround(creal(pa[k]) / (double)L);", "c[k] = (int64_t)(creal(pa[k]) / (double)L);"),
    ("modular evaluation: off by one",
     "acc = (acc * tt + ar) % p;", "acc = (acc * tt + ar + 1) % p;"),
    ("convolution: filter index shifted",
     "cplx term = xc[i] * hc[k - i];", "cplx term = xc[i] * hc[k - i > 0 ? k - i - 1 : 0];"),
    ("real transform: the last half-spectrum bin not written",
     "memcpy(X, Z, sizeof(cplx) * (size_t)(n / 2 + 1));", "memcpy(X, Z, sizeof(cplx) * (size_t)(n / 2));"),
    ("real inverse: mirrored bins not conjugated",
     "Y[k] = 2 * k <= n ? half[k] : conj(half[n - k]);", "Y[k] = 2 * k <= n ? half[k] : half[n - k];"),
    ("real inverse: 1/N dropped",
     "x[i] = creal(y[i]) / (double)n;", "x[i] = creal(y[i]);"),
]


def _build(src_text, td, name):
    path = os.path.join(td, name + ".c")
    with open(path, "w") as f:
        f.write(src_text)
    lib = os.path.join(td, name + ".so")
    subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-o", lib, path, "-lm"])
    return lib


def _pins_pass(lib):
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=lib)
    res = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
                          "-x", "-q", "-p", "no:cacheprovider"],
                         env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    return res.returncode == 0


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unmutated_copy_passes(source):
    with tempfile.TemporaryDirectory() as td:
        assert _pins_pass(_build(source, td, "clean"))


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(source, name, old, new):
    assert source.count(old) >= 1, f"mutation site not found: {name}"
    with tempfile.TemporaryDirectory() as td:
        lib = _build(source.replace(old, new), td, "mutant")
        assert not _pins_pass(lib), f"no pin caught: {name}"
