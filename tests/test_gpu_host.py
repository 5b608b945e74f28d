"""Host-buffer pipelines through the C ABI: fft_convolve_host and
polymul_batched_host stream chunks of rows through the device (uploads,
compute and downloads overlapping); results against the oracle, with chunk
sizes that do not divide the batch."""
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


def sh():
    return int(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("kind,per_row,nx,nh,batch,chunk", [
    (1, 0, 3072, 1025, 37, 8), (1, 1, 300, 57, 10, 3), (0, 0, 500, 200, 9, 4),
    (0, 1, 1000, 33, 5, 2), (1, 0, 20000, 7000, 3, 1)])
def test_convolve_host(fg, kind, per_row, nx, nh, batch, chunk):
    if kind == 1:
        x = workloads.normal_real((batch, nx), 9800 + nx, np.float32)
        h = workloads.normal_real((batch if per_row else 1, nh), 9801, np.float32)
        ydt = torch.float32
    else:
        x = workloads.normal_complex((batch, nx), 9800 + nx, np.complex64)
        h = workloads.normal_complex((batch if per_row else 1, nh), 9801, np.complex64)
        ydt = torch.complex64
    ny = nx + nh - 1
    hx = torch.from_numpy(x).pin_memory()
    hy = torch.empty(batch, ny, dtype=ydt).pin_memory()
    hd = torch.from_numpy(h).cuda()
    dx = torch.empty(batch, nx, dtype=hx.dtype, device="cuda")
    dy = torch.empty(batch, ny, dtype=ydt, device="cuda")
    rc = fg.fft_convolve_host(hx.data_ptr(), nx, hd.data_ptr(), nh, hy.data_ptr(), batch, per_row,
                              kind, 0, dx.data_ptr(), dy.data_ptr(), chunk, sh())
    torch.cuda.synchronize()
    assert rc == 0, fg.fft_status_string(rc)
    got = hy.numpy().astype(np.complex128)
    L = 1 << (ny - 1).bit_length()
    for r in range(batch):
        ref = oracle.convolve(x[r].astype(np.complex128),
                              h[r if per_row else 0].astype(np.complex128))
        assert np.linalg.norm(got[r] - ref) / np.linalg.norm(ref) <= 1e-5 * int(np.log2(L))


@pytest.mark.parametrize("na,nb,batch,chunk", [(1000, 3000, 7, 3), (1 << 12, 1 << 12, 4, 4),
                                               (5, 7, 9, 2)])
def test_polymul_host(fg, na, nb, batch, chunk):
    g = workloads.generator(9900 + na)
    a = g.integers(0, 10, size=(batch, na), dtype=np.int64)
    b = g.integers(0, 10, size=(batch, nb), dtype=np.int64)
    ha, hb = torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory()
    hc = torch.empty(batch, na + nb - 1, dtype=torch.int64).pin_memory()
    da = torch.empty_like(ha, device="cuda")
    db = torch.empty_like(hb, device="cuda")
    dc = torch.empty_like(hc, device="cuda")
    rc = fg.polymul_batched_host(ha.data_ptr(), na, hb.data_ptr(), nb, hc.data_ptr(), batch,
                                 da.data_ptr(), db.data_ptr(), dc.data_ptr(), chunk, sh())
    torch.cuda.synchronize()
    assert rc == 0, fg.fft_status_string(rc)
    for r in range(batch):
        assert np.array_equal(hc[r].numpy(), oracle.polymul_schoolbook(a[r], b[r]))


@pytest.mark.parametrize("kind", ["c2c", "real_fwd", "real_inv", "nd"])
def test_exec_host_single_shot(fg, kind):
    # fft_exec_host: upload, transform and download on one stream, with the
    # plan's own input and output sizes (real plans differ).
    if kind == "c2c":
        n, batch = 3000, 4
        p = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_C2C_F32)
        x = workloads.normal_complex((batch, n), 9950, np.complex64)
        ref = np.stack([oracle.dft(r.astype(np.complex128)) for r in x])
        out_shape, out_dt = (batch, n), torch.complex64
    elif kind == "real_fwd":
        n, batch = 1000, 3
        p = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_REAL_F32)
        x = workloads.normal_real((batch, n), 9951, np.float32)
        ref = oracle.rfft(x.astype(np.float64))
        out_shape, out_dt = (batch, n // 2 + 1), torch.complex64
    elif kind == "real_inv":
        n, batch = 1000, 3
        p = fg.Plan(n, batch, 1, fg.FFT_INVERSE, fg.FFT_REAL_F32)
        g = workloads.generator(9952)
        x = (g.standard_normal((batch, n // 2 + 1)) +
             1j * g.standard_normal((batch, n // 2 + 1))).astype(np.complex64)
        ref = oracle.irfft(x.astype(np.complex128), n)
        out_shape, out_dt = (batch, n), torch.float32
    else:
        shape, batch = (30, 64), 2
        p = fg.Plan(0, batch, direction=fg.FFT_FORWARD, dtype=fg.FFT_C2C_F32, shape=shape)
        x = workloads.normal_complex((batch,) + shape, 9953, np.complex64)
        ref = oracle.fftn(x.astype(np.complex128), 2).reshape(batch, -1)
        out_shape, out_dt = (batch,) + shape, torch.complex64
    hin = torch.from_numpy(x).pin_memory()
    hout = torch.empty(out_shape, dtype=out_dt).pin_memory()
    din = torch.empty_like(hin, device="cuda")
    dout = torch.empty(out_shape, dtype=out_dt, device="cuda")
    p.exec_host(hin, hout, din, dout)
    torch.cuda.synchronize()
    got = hout.numpy().reshape(ref.shape[0], -1).astype(np.complex128)
    want = ref.reshape(ref.shape[0], -1)
    err = np.linalg.norm(got - want, axis=1) / np.linalg.norm(want, axis=1)
    assert err.max() <= 1e-5 * 13
    p.close()
