"""Seeded random sweep over the plan kinds: random lengths (powers of two,
smooth, prime and other), batches, precisions and directions for 1D complex,
real, 2D / 3D, convolution and polymul, each checked against the oracle.
Sizes are drawn so that the oracle finishes in seconds."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = 240
TOL = {0: 1e-5, 1: 1e-13}
CT = {0: np.complex64, 1: np.complex128}
RT = {0: np.float32, 1: np.float64}


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


def draw_length(g, cap_other=3000, cap_pow2=1 << 16):
    kind = g.integers(0, 4)
    if kind == 0:
        return int(1 << g.integers(0, cap_pow2.bit_length()))
    if kind == 1:   # smooth: 2^a 3^b 5^c 7^d 11^e 13^f
        n = 1
        for f, e in ((2, 6), (3, 4), (5, 3), (7, 2), (11, 1), (13, 1)):
            n *= f ** int(g.integers(0, e + 1))
        return int(min(n, cap_other)) if n <= cap_other else 3 * 5 * 7
    return int(g.integers(1, cap_other + 1))


def tol_for(dtype, n):
    """The relative-L2 bound of a transform of n points: 1e-5 log2(n) (fp32),
    1e-13 log2(n) (fp64), whichever algorithm the plan takes for n."""
    return TOL[dtype] * max(1, int(np.log2(max(n, 1))))


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz(fg, case):
    g = workloads.generator(20000 + case)
    what = case % 5
    dtype = int(g.integers(0, 2))
    direction = -1 if g.integers(0, 2) == 0 else 1
    batch = int(g.integers(1, 6))
    if what == 0:                                   # 1D complex, any length
        n = draw_length(g)
        x = workloads.normal_complex((batch, n), 21000 + case, CT[dtype])
        p = fg.Plan(n, batch, 1, direction, dtype)
        y = p.exec(torch.from_numpy(x).cuda())
        torch.cuda.synchronize()
        p.close()
        ref = np.stack([oracle.dft(r.astype(np.complex128), direction) if n & (n - 1)
                        else (oracle.fft(r.astype(np.complex128)) if direction < 0
                              else oracle.ifft(r.astype(np.complex128))) for r in x])
        assert rel_rows(y.cpu().numpy(), ref).max() <= tol_for(dtype, n), (n, batch, dtype)
    elif what == 1:                                 # real, any length
        n = draw_length(g)
        if direction < 0:
            x = workloads.normal_real((batch, n), 22000 + case, RT[dtype])
            X = fg.rfft(torch.from_numpy(x).cuda())
            torch.cuda.synchronize()
            ref = oracle.rfft(x.astype(np.float64))
            assert rel_rows(X.cpu().numpy(), ref).max() <= tol_for(dtype, n), (n, dtype)
        else:
            X = (g.standard_normal((batch, n // 2 + 1)) +
                 1j * g.standard_normal((batch, n // 2 + 1))).astype(CT[dtype])
            y = fg.irfft(torch.from_numpy(X).cuda(), n)
            torch.cuda.synchronize()
            ref = oracle.irfft(X.astype(np.complex128), n)
            assert rel_rows(y.cpu().numpy(), ref).max() <= tol_for(dtype, n), (n, dtype)
    elif what == 2:                                 # 2D / 3D, any sides
        rank = int(g.integers(2, 4))
        cap_o, cap_p = (150, 256) if rank == 2 else (60, 64)
        shape = tuple(int(v) for v in (draw_length(g, cap_other=cap_o, cap_pow2=cap_p)
                                       for _ in range(rank)))
        x = workloads.normal_complex((batch,) + shape, 23000 + case, CT[dtype])
        p = fg.Plan(0, batch, direction=direction, dtype=dtype, shape=shape)
        y = p.exec(torch.from_numpy(x).cuda())
        torch.cuda.synchronize()
        p.close()
        ref = oracle.fftn(x.astype(np.complex128), rank, direction)
        assert rel_rows(y.cpu().numpy(), ref).max() <= tol_for(dtype, int(np.prod(shape))), \
            (shape, dtype)
    elif what == 3:                                 # convolution
        nx, nh = int(g.integers(1, 3000)), int(g.integers(1, 1500))
        real = bool(g.integers(0, 2))
        per_row = int(g.integers(0, 2))
        nf = batch if per_row else 1
        if real:
            x = workloads.normal_real((batch, nx), 24000 + case, RT[dtype])
            h = workloads.normal_real((nf, nh), 24500 + case, RT[dtype])
        else:
            x = workloads.normal_complex((batch, nx), 24000 + case, CT[dtype])
            h = workloads.normal_complex((nf, nh), 24500 + case, CT[dtype])
        hh = torch.from_numpy(h if per_row else h[0]).cuda()
        y = fg.convolve(torch.from_numpy(x).cuda(), hh)
        torch.cuda.synchronize()
        ref = oracle.convolve(x.astype(np.complex128), (h if per_row else h[0]).astype(np.complex128))
        L = 1 << max(1, (nx + nh - 2).bit_length())
        assert rel_rows(y.cpu().numpy(), ref).max() <= TOL[dtype] * max(1, int(np.log2(L))), \
            (nx, nh, real, per_row, dtype)
    else:                                           # polymul, exact
        na, nb = int(g.integers(1, 5000)), int(g.integers(1, 5000))
        a = g.integers(-9, 10, size=(batch, na), dtype=np.int64)
        b = g.integers(-9, 10, size=(batch, nb), dtype=np.int64)
        c = fg.polymul_tensors(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
        torch.cuda.synchronize()
        for r in range(batch):
            assert np.array_equal(c[r].cpu().numpy(), oracle.polymul_schoolbook(a[r], b[r])), (na, nb)
