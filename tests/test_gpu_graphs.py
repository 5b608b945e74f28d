"""The library's enqueue-only entry points inside CUDA graphs: fft_exec of
every plan kind, fft_convolve and polymul_batched (stream-ordered scratch
becomes graph memory nodes) are captured once with torch.cuda.graph and
replayed on new data in the same buffers; each replay matches the oracle."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg(fg_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fg_lib


def rel_rows(y, ref):
    y = np.asarray(y).reshape(ref.shape[0], -1).astype(np.complex128)
    ref = np.asarray(ref).reshape(ref.shape[0], -1).astype(np.complex128)
    return np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)


def sh():
    return int(torch.cuda.current_stream().cuda_stream)


def capture(fn):
    """Warm up fn once on a side stream, then capture it into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("n,batch", [(4096, 64), (1 << 18, 2), (3000, 8), (10007, 2)])
def test_graph_forward_inverse(fg, n, batch):
    pf = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_C2C_F32)
    pi = fg.Plan(n, batch, 1, fg.FFT_INVERSE, fg.FFT_C2C_F32)
    x = torch.empty(batch, n, dtype=torch.complex64, device="cuda")
    y, z = torch.empty_like(x), torch.empty_like(x)

    def step():
        assert fg.fft_exec(pf.handle, x.data_ptr(), y.data_ptr(), sh()) == 0
        assert fg.fft_exec(pi.handle, y.data_ptr(), z.data_ptr(), sh()) == 0
    x.copy_(torch.from_numpy(workloads.normal_complex((batch, n), 9500, np.complex64)))
    g = capture(step)
    for seed in (9501, 9502):
        h = workloads.normal_complex((batch, n), seed, np.complex64)
        x.copy_(torch.from_numpy(h))
        g.replay()
        torch.cuda.synchronize()
        rows = [0, batch - 1]
        pow2 = n & (n - 1) == 0
        ref = np.stack([(oracle.fft if pow2 else oracle.dft)(h[r].astype(np.complex128))
                        for r in rows])
        bl = n if pow2 or n == 3000 else 1 << (2 * n - 2).bit_length()
        tol = 1e-5 * int(np.log2(bl))
        assert rel_rows(y.cpu().numpy()[rows], ref).max() <= tol
        assert rel_rows(z.cpu().numpy(), h).max() <= 2 * tol
    pf.close()
    pi.close()


def test_graph_real_and_nd(fg):
    n, batch = 1 << 16, 3                       # real, split around a multi-pass plan
    pf = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_REAL_F32)
    p3 = fg.Plan(0, 2, direction=fg.FFT_FORWARD, dtype=fg.FFT_C2C_F32, shape=(16, 32, 64))
    x = torch.empty(batch, n, dtype=torch.float32, device="cuda")
    X = torch.empty(batch, n // 2 + 1, dtype=torch.complex64, device="cuda")
    v = torch.empty(2, 16, 32, 64, dtype=torch.complex64, device="cuda")
    V = torch.empty_like(v)

    def step():
        assert fg.fft_exec(pf.handle, x.data_ptr(), X.data_ptr(), sh()) == 0
        assert fg.fft_exec(p3.handle, v.data_ptr(), V.data_ptr(), sh()) == 0
    g = capture(step)
    xs = workloads.normal_real((batch, n), 9600, np.float32)
    vs = workloads.normal_complex((2, 16, 32, 64), 9601, np.complex64)
    x.copy_(torch.from_numpy(xs))
    v.copy_(torch.from_numpy(vs))
    g.replay()
    torch.cuda.synchronize()
    assert rel_rows(X.cpu().numpy(), oracle.rfft(xs.astype(np.float64))).max() <= 1e-5 * 15
    ref = oracle.fftn(vs.astype(np.complex128), 3)
    assert rel_rows(V.cpu().numpy(), ref).max() <= 1e-5 * 15
    pf.close()
    p3.close()


def test_graph_polymul_and_convolve(fg):
    # Both allocate their scratch stream-ordered: inside a graph these are
    # memory nodes of the graph.
    na, nb, batch = 1000, 3000, 2
    a = torch.empty(batch, na, dtype=torch.int64, device="cuda")
    b = torch.empty(batch, nb, dtype=torch.int64, device="cuda")
    c = torch.empty(batch, na + nb - 1, dtype=torch.int64, device="cuda")
    nx, nh = 3072, 1025
    xs = torch.empty(4, nx, dtype=torch.float32, device="cuda")
    hs = torch.empty(nh, dtype=torch.float32, device="cuda")
    ys = torch.empty(4, nx + nh - 1, dtype=torch.float32, device="cuda")

    def step():
        assert fg.polymul_batched(a.data_ptr(), na, b.data_ptr(), nb, c.data_ptr(), batch,
                                  sh()) == 0
        assert fg.fft_convolve(xs.data_ptr(), nx, hs.data_ptr(), nh, ys.data_ptr(), 4, 0,
                               fg.FFT_CONV_REAL, fg.FFT_C2C_F32, sh()) == 0
    gen = workloads.generator(9700)
    a.copy_(torch.from_numpy(gen.integers(0, 10, size=(batch, na), dtype=np.int64)))
    b.copy_(torch.from_numpy(gen.integers(0, 10, size=(batch, nb), dtype=np.int64)))
    g = capture(step)
    for seed in (9701, 9702):
        gen = workloads.generator(seed)
        ah = gen.integers(0, 10, size=(batch, na), dtype=np.int64)
        bh = gen.integers(0, 10, size=(batch, nb), dtype=np.int64)
        xh, hh = workloads.conv_signals(4, nx, nh, seed)
        a.copy_(torch.from_numpy(ah))
        b.copy_(torch.from_numpy(bh))
        xs.copy_(torch.from_numpy(xh))
        hs.copy_(torch.from_numpy(hh))
        g.replay()
        torch.cuda.synchronize()
        for r in range(batch):
            assert np.array_equal(c[r].cpu().numpy(), oracle.polymul_schoolbook(ah[r], bh[r]))
        ref = oracle.convolve(xh.astype(np.complex128), hh.astype(np.complex128))
        assert rel_rows(ys.cpu().numpy(), ref).max() <= 1e-5 * 12
