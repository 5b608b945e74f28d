"""GPU parity of the transforms of real sequences (FFT_REAL_F32 / _F64)
through the C ABI against the fp64 oracle (oracle.rfft / oracle.irfft) on
the same seeded samples.

Forward: the half spectrum of each row; inverse: real rows from arbitrary
half spectra (random bins, including imaginary parts at DC and Nyquist that
the definition drops), so the inverse is checked on its own and not only as
a round trip.  Tolerance: relative L2 per row <= 1e-5 log2(n) (fp32),
1e-13 log2(n) (fp64); Bluestein-backed lengths use the convolution length.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

R32, R64 = 2, 3
TOL = {R32: 1e-5, R64: 1e-13}
RT = {R32: np.float32, R64: np.float64}
CT = {R32: np.complex64, R64: np.complex128}


@pytest.fixture(scope="module")
def fg(fg_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fg_lib


def rel_rows(y, ref):
    y = np.asarray(y).reshape(ref.shape[0], -1).astype(np.complex128)
    ref = np.asarray(ref).reshape(ref.shape[0], -1).astype(np.complex128)
    den = np.linalg.norm(ref, axis=1)
    den[den == 0] = 1
    return np.linalg.norm(y - ref, axis=1) / den


def work_len(n):
    """Length of the transform that carries most of the error: n/2 for even
    n through a power-of-two path, the Bluestein length otherwise."""
    m = n // 2 if n % 2 == 0 else n
    if m & (m - 1) == 0 or m <= 64:
        return max(2, n)
    return 1 << (2 * m - 2).bit_length()


def tol(dtype, n):
    return TOL[dtype] * max(1, int(np.log2(work_len(n))))


def forward(fg, x, dtype):
    batch, n = x.shape
    p = fg.Plan(n, batch, 1, fg.FFT_FORWARD, dtype)
    X = p.exec(torch.from_numpy(np.ascontiguousarray(x)).cuda())
    torch.cuda.synchronize()
    kernels = p.num_kernels
    p.close()
    return X.cpu().numpy(), kernels


def inverse(fg, X, n, dtype):
    batch = X.shape[0]
    p = fg.Plan(n, batch, 1, fg.FFT_INVERSE, dtype)
    y = p.exec(torch.from_numpy(np.ascontiguousarray(X)).cuda())
    torch.cuda.synchronize()
    p.close()
    return y.cpu().numpy()


def random_half_spectrum(batch, n, seed, dtype):
    g = workloads.generator(seed)
    shape = (batch, n // 2 + 1)
    X = g.standard_normal(size=shape) + 1j * g.standard_normal(size=shape)
    return X.astype(CT[dtype])


def check_both(fg, n, batch, dtype, seed):
    x = workloads.normal_real((batch, n), seed, RT[dtype])
    X, kernels = forward(fg, x, dtype)
    assert X.shape == (batch, n // 2 + 1) and X.dtype == CT[dtype]
    assert rel_rows(X, oracle.rfft(x.astype(np.float64))).max() <= tol(dtype, n)
    S = random_half_spectrum(batch, n, seed + 1, dtype)
    y = inverse(fg, S, n, dtype)
    assert y.shape == (batch, n) and y.dtype == RT[dtype]
    assert rel_rows(y, oracle.irfft(S.astype(np.complex128), n)).max() <= tol(dtype, n)
    return kernels


# --- n = 2H, H a power of two on chip: one kernel each way ------------------------

@pytest.mark.parametrize("dtype", [R32, R64])
@pytest.mark.parametrize("logn", list(range(1, 16)))
def test_real_on_chip(fg, dtype, logn):
    if dtype == R64 and logn > 14:
        pytest.skip("fp64 on-chip limit is H = 2^13")
    n = 1 << logn
    batch = 5 if n >= 512 else 37   # ragged against the rows per block
    assert check_both(fg, n, batch, dtype, 7000 + logn) == 1


# --- other even n: complex plan of length n/2 + split kernel over HBM ---------------

@pytest.mark.parametrize("dtype,n", [(R32, 1 << 16), (R32, 1 << 18), (R64, 1 << 15), (R64, 1 << 17),
                                     (R32, 6), (R32, 100), (R32, 3000), (R64, 130), (R64, 2 * 4097),
                                     (R32, 2 * 10007)])
def test_real_even_split(fg, dtype, n):
    assert check_both(fg, n, 3, dtype, 7100 + n % 1000) >= 2


# --- odd n: complex plan of length n ---------------------------------------------

@pytest.mark.parametrize("dtype,n", [(R32, 1), (R64, 1), (R32, 3), (R32, 63), (R64, 65),
                                     (R32, 1001), (R64, 3001)])
def test_real_odd(fg, dtype, n):
    assert check_both(fg, n, 4, dtype, 7200 + n) >= 3


def test_real_round_trip_and_hermitian_input(fg):
    # The round trip returns the samples; a spectrum taken from the forward
    # transform has real DC and Nyquist bins, so nothing is dropped.
    n, batch = 4096, 9
    x = workloads.normal_real((batch, n), 7300, np.float32)
    X, _ = forward(fg, x, R32)
    assert np.abs(X[:, 0].imag).max() == 0 and np.abs(X[:, -1].imag).max() == 0
    y = inverse(fg, X, n, R32)
    assert rel_rows(y, x).max() <= 2 * tol(R32, n)


def test_real_matches_complex_transform(fg):
    # The half spectrum equals the first n/2 + 1 bins of the complex
    # transform of the same samples (the library's own complex path).
    n, batch = 1 << 12, 6
    x = workloads.normal_real((batch, n), 7400, np.float64)
    X, _ = forward(fg, x, R64)
    p = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_C2C_F64)
    Z = p.exec(torch.from_numpy(x.astype(np.complex128)).cuda())
    torch.cuda.synchronize()
    p.close()
    assert rel_rows(X, Z.cpu().numpy()[:, : n // 2 + 1]).max() <= tol(R64, n)


@pytest.mark.parametrize("n,chunk", [(8192, 4), (3000, 2), (1 << 16, 2)])
def test_real_host_chain(fg, n, chunk):
    # R2C then C2R through the chunked host pipeline (different sizes in and
    # out of each plan).
    batch = 6
    x = workloads.normal_real((batch, n), 7500 + n % 1000, np.float32)
    pf = fg.Plan(n, batch, 1, fg.FFT_FORWARD, R32)
    pi = fg.Plan(n, batch, 1, fg.FFT_INVERSE, R32)
    h_in = torch.from_numpy(x).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    da = torch.empty(batch * n, dtype=torch.float32, device="cuda")
    db = torch.empty(batch * (n // 2 + 1), dtype=torch.complex64, device="cuda")
    pf.chain_host([pi], h_in, h_out, da, db, chunk)
    torch.cuda.synchronize()
    assert rel_rows(h_out.numpy(), x).max() <= 2 * tol(R32, n)
    pf.close()
    pi.close()


def test_real_chain_rejects_misaligned_chunks(fg):
    # n = 6: 24-byte sample rows; chunks of one row would start off 16 bytes.
    pf = fg.Plan(6, 4, 1, fg.FFT_FORWARD, R32)
    pi = fg.Plan(6, 4, 1, fg.FFT_INVERSE, R32)
    h = torch.zeros(24, dtype=torch.float32).pin_memory()
    da = torch.empty(24, dtype=torch.float32, device="cuda")
    db = torch.empty(16, dtype=torch.complex64, device="cuda")
    rc = fg.fft_exec_host_chain([pf.handle, pi.handle], 2, h.data_ptr(), h.data_ptr(),
                                da.data_ptr(), db.data_ptr(), 1, None)
    assert rc == fg.FFT_ERR_MISALIGNED
    pf.close()
    pi.close()


def test_rfft_irfft_helpers(fg):
    x = workloads.normal_real((2, 3, 512), 7600, np.float32)
    X = fg.rfft(torch.from_numpy(x).cuda())
    assert tuple(X.shape) == (2, 3, 257)
    ref = oracle.rfft(x.astype(np.float64).reshape(6, 512))
    assert rel_rows(X.cpu().numpy().reshape(6, 257), ref).max() <= tol(R32, 512)
    y = fg.irfft(X, 512)
    assert tuple(y.shape) == (2, 3, 512)
    assert rel_rows(y.cpu().numpy().reshape(6, 512), x.reshape(6, 512)).max() <= 2 * tol(R32, 512)
