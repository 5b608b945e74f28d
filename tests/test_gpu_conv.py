"""GPU parity of the signal convolution (fft_convolve) against the oracle's
direct sum y_k = sum_i x_i h_{k-i}.

Covers complex and real samples, fp32 and fp64, one shared filter and one
filter per row, the fused on-chip path (L <= 2^14 fp32 / 2^13 fp64), the
multi-pass path, ragged batches (an odd number of real rows travels in pairs
with one half-empty pair) and the degenerate lengths.  Tolerance: relative
L2 error per row <= 1e-5 * log2(L) (fp32) / 1e-13 * log2(L) (fp64).
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TORCH = {("c", 0): torch.complex64, ("c", 1): torch.complex128,
         ("r", 0): torch.float32, ("r", 1): torch.float64}
NP = {("c", 0): np.complex64, ("c", 1): np.complex128, ("r", 0): np.float32, ("r", 1): np.float64}


@pytest.fixture(scope="module")
def fg(fg_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fg_lib


def make(kind, dtype, shape, seed):
    z = workloads.normal_complex(shape, seed, np.complex128)
    return (z if kind == "c" else z.real).astype(NP[(kind, dtype)])


def check(fg, kind, dtype, nx, nh, batch, per_row, seed=0):
    x = make(kind, dtype, (batch, nx), 100 + seed)
    h = make(kind, dtype, (batch, nh) if per_row else (nh,), 200 + seed)
    y = fg.convolve(torch.from_numpy(x).cuda(), torch.from_numpy(h).cuda())
    torch.cuda.synchronize()
    y = y.cpu().numpy().astype(np.complex128)
    ref = oracle.convolve(x.astype(np.complex128), h.astype(np.complex128))
    ny = nx + nh - 1
    L = 1 << max(1, (ny - 1).bit_length())
    tol = (1e-5 if dtype == 0 else 1e-13) * max(1, L.bit_length() - 1)
    err = np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert y.shape == (batch, ny)
    assert err.max() <= tol, (err.max(), tol)
    if kind == "r":
        assert np.max(np.abs(ref.imag)) < 1e-9


@pytest.mark.parametrize("kind", ["c", "r"])
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("per_row", [0, 1])
@pytest.mark.parametrize("nx,nh,batch", [(1, 1, 1), (5, 3, 3), (1000, 31, 5), (3072, 1025, 3),
                                         (200, 1800, 2)])
def test_fused_on_chip(fg, kind, dtype, per_row, nx, nh, batch):
    check(fg, kind, dtype, nx, nh, batch, per_row)


@pytest.mark.parametrize("kind,dtype,nx,nh", [("c", 0, 9000, 7385),     # L = 2^14, fp32 on chip
                                              ("c", 1, 5000, 3193)])    # L = 2^13, fp64 on chip
def test_largest_on_chip(fg, kind, dtype, nx, nh):
    check(fg, kind, dtype, nx, nh, 2, 0)


@pytest.mark.parametrize("kind,dtype,nx,nh,batch,per_row", [
    ("c", 0, 20000, 13000, 2, 0),   # L = 2^16 fp32: passes 8, 8
    ("r", 0, 30000, 9000, 3, 0),    # L = 2^16, real pairs (one half-empty)
    ("r", 0, 12000, 5000, 2, 1),    # L = 2^15, real rows with their own filters
    ("c", 1, 9000, 8000, 1, 1),     # L = 2^15 fp64: passes 8, 7
])
def test_multipass(fg, kind, dtype, nx, nh, batch, per_row):
    check(fg, kind, dtype, nx, nh, batch, per_row, seed=nx)


def test_delta_filter_and_shift(fg):
    x = workloads.normal_complex((4, 777), 9).astype(np.complex64)
    d = np.zeros(9, np.complex64)
    d[3] = 1
    y = fg.convolve(torch.from_numpy(x).cuda(), torch.from_numpy(d).cuda()).cpu().numpy()
    assert np.max(np.abs(y[:, 3:780] - x)) < 1e-5
    assert np.max(np.abs(y[:, :3])) < 1e-5 and np.max(np.abs(y[:, 780:])) < 1e-5


def test_argument_checks(fg):
    st = int(torch.cuda.current_stream().cuda_stream)
    buf = torch.zeros(64, dtype=torch.complex64, device="cuda")
    p = buf.data_ptr()
    assert fg.fft_convolve(p, 0, p, 4, p, 1, 0, 0, 0, st) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_convolve(p, 4, p, 4, p, 1, 2, 0, 0, st) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_convolve(p, 4, p, 4, p, 1, 0, 5, 0, st) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_convolve(p + 4, 4, p, 4, p, 1, 0, 0, 0, st) == fg.FFT_ERR_MISALIGNED
    assert fg.fft_convolve(p, 1 << 27, p, 1 << 27, p, 1, 0, 0, 0, st) == fg.FFT_ERR_UNSUPPORTED
    assert fg.fft_convolve_num_kernels(3072, 1025, 8, 0, 1, 0) == 2
