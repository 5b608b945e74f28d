"""Guard bands around every buffer a kernel touches: each input and output
lives inside a larger allocation whose margins hold a byte pattern; after
the call the margins must be unchanged (no write outside the output, none at
all into the input) for every kind of plan, on ragged sizes.  Also the
allocation-failure path: a plan whose workspace cannot be allocated returns
FFT_ERR_ALLOC and leaves the device usable."""
import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 4096        # bytes on each side (keeps the data 16-byte aligned)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def fg(fg_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fg_lib


class Guarded:
    """`nbytes` of device memory at .ptr with patterned margins."""

    def __init__(self, data: np.ndarray = None, nbytes: int = None):
        raw = data.view(np.uint8).reshape(-1) if data is not None else None
        self.nbytes = raw.size if raw is not None else nbytes
        self.buf = torch.full((self.nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        if raw is not None:
            self.buf[GUARD:GUARD + self.nbytes] = torch.from_numpy(raw.copy()).cuda()
        self.initial = self.buf.cpu().numpy().copy()
        self.ptr = self.buf.data_ptr() + GUARD

    def margins_intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == PATTERN).all() and (b[GUARD + self.nbytes:] == PATTERN).all())

    def unchanged(self) -> bool:
        return bool((self.buf.cpu().numpy() == self.initial).all())


def stream():
    return int(torch.cuda.current_stream().cuda_stream)


def run_guarded_plan(fg, plan, in_bytes_data, out_nbytes):
    gi = Guarded(in_bytes_data)
    go = Guarded(nbytes=out_nbytes)
    rc = fg.fft_exec(plan.handle, gi.ptr, go.ptr, stream())
    torch.cuda.synchronize()
    assert rc == 0, fg.fft_status_string(rc)
    assert gi.unchanged(), "input or its margins modified"
    assert go.margins_intact(), "write outside the output"


C2C = [  # (n, batch, dtype)
    (64, 37, 0), (4096, 3, 0), (8192, 2, 1), (1 << 16, 3, 0), (1 << 15, 2, 1),   # pow2 rows / passes
    (12, 37, 0), (63, 5, 1),                                                    # direct DFT
    (100, 37, 0), (3000, 3, 0), (6144, 2, 1),                                   # mixed radix
    (1009, 3, 0), (10007, 2, 0), (4091, 2, 1),                                  # Bluestein
]


@pytest.mark.parametrize("n,batch,dtype", C2C)
@pytest.mark.parametrize("direction", [-1, 1])
def test_c2c_guards(fg, n, batch, dtype, direction):
    np_t = np.complex64 if dtype == 0 else np.complex128
    x = workloads.normal_complex((batch, n), 9000 + n, np_t)
    p = fg.Plan(n, batch, 1, direction, dtype)
    run_guarded_plan(fg, p, x, x.nbytes)
    p.close()


@pytest.mark.parametrize("shape,batch", [((64, 64), 3), ((16, 32), 5), ((4, 16, 32), 2),
                                         ((2, 1, 256), 3), ((30, 50), 3), ((3, 5, 7), 2),
                                         ((1 << 15, 4), 1), ((2048, 256), 2), ((2, 1024, 256), 1)])
def test_nd_guards(fg, shape, batch):
    x = workloads.normal_complex((batch,) + shape, 9100, np.complex64)
    for direction in (-1, 1):
        p = fg.Plan(0, batch, direction=direction, dtype=0, shape=shape)
        run_guarded_plan(fg, p, x, x.nbytes)
        p.close()


@pytest.mark.parametrize("n,batch,dtype", [(2, 37, 2), (4096, 5, 2), (8192, 3, 3), (6, 7, 2),
                                           (3000, 3, 2), (1 << 16, 2, 2), (63, 3, 2), (1, 5, 3)])
def test_real_guards(fg, n, batch, dtype):
    rt, ct = (np.float32, np.complex64) if dtype == 2 else (np.float64, np.complex128)
    x = workloads.normal_real((batch, n), 9200 + n, rt)
    bins = np.empty((batch, n // 2 + 1), ct)
    pf = fg.Plan(n, batch, 1, -1, dtype)
    run_guarded_plan(fg, pf, x, bins.nbytes)
    pf.close()
    g = workloads.generator(9300 + n)
    X = (g.standard_normal(bins.shape) + 1j * g.standard_normal(bins.shape)).astype(ct)
    pi = fg.Plan(n, batch, 1, 1, dtype)
    run_guarded_plan(fg, pi, X, x.nbytes)
    pi.close()


@pytest.mark.parametrize("nx,nh,batch,per_row,kind", [(3072, 1025, 5, 0, 1), (100, 7, 9, 1, 1),
                                                      (300, 50, 3, 0, 0), (40000, 30000, 1, 0, 1)])
def test_convolve_guards(fg, nx, nh, batch, per_row, kind):
    real = kind == 1
    if real:
        x = workloads.normal_real((batch, nx), 9400, np.float32)
        h = workloads.normal_real((batch if per_row else 1, nh), 9401, np.float32)
        out_bytes = batch * (nx + nh - 1) * 4
    else:
        x = workloads.normal_complex((batch, nx), 9400, np.complex64)
        h = workloads.normal_complex((batch if per_row else 1, nh), 9401, np.complex64)
        out_bytes = batch * (nx + nh - 1) * 8
    gx, gh, gy = Guarded(x), Guarded(h), Guarded(nbytes=out_bytes)
    rc = fg.fft_convolve(gx.ptr, nx, gh.ptr, nh, gy.ptr, batch, per_row, kind, 0, stream())
    torch.cuda.synchronize()
    assert rc == 0, fg.fft_status_string(rc)
    assert gx.unchanged() and gh.unchanged() and gy.margins_intact()


@pytest.mark.parametrize("na,nb,batch", [(5, 7, 3), (1000, 3000, 2), (1 << 12, 1 << 12, 2)])
def test_polymul_guards(fg, na, nb, batch):
    g = workloads.generator(na + nb)
    a = g.integers(0, 10, size=(batch, na), dtype=np.int64)
    b = g.integers(0, 10, size=(batch, nb), dtype=np.int64)
    ga, gb, gc = Guarded(a), Guarded(b), Guarded(nbytes=batch * (na + nb - 1) * 8)
    rc = fg.polymul_batched(ga.ptr, na, gb.ptr, nb, gc.ptr, batch, stream())
    torch.cuda.synchronize()
    assert rc == 0
    assert ga.unchanged() and gb.unchanged() and gc.margins_intact()


@pytest.mark.parametrize("n,batch,dtype", [(1 << 20, 1 << 19, 0), (1 << 17, 1 << 22, 2),
                                           (10007, 1 << 24, 0)])
def test_workspace_allocation_failure(fg, n, batch, dtype):
    # Workspaces of several TB cannot be allocated: the plan reports ALLOC,
    # and the device keeps working afterwards.
    h = fg._lib.fft_plan_create(n, batch, 1, -1, dtype)
    assert not h
    assert fg.fft_last_status() == fg.FFT_ERR_ALLOC
    x = torch.ones(4, 64, dtype=torch.complex64, device="cuda")
    y = fg.fft(x)
    torch.cuda.synchronize()
    assert torch.allclose(y[:, 0].real, torch.full((4,), 64.0, device="cuda"))
