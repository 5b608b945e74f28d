"""GPU parity at the benchmark sizes, in the launch configuration bench.py
times (out-of-place plans over the whole batch), on outputs the oracle can
compute one by one, plus properties that hold at any size.

* 16384 x 4096 fp32: 48 sampled transforms against the recursive CT; the
  inverse returns the input for every transform.
* one 2^26 fp32 transform (16 tones + noise): the whole vector against the
  oracle's recursive Cooley-Tukey (relative L2 error), the 16 tone bins also
  against the direct DFT of those bins; Parseval and the inverse round trip
  over the whole vector.
* 8 images of 2048 x 2048 fp32: images 0 and 7 against the oracle's 2D
  transform; the inverse round trip for all 8.
* 64 polynomial pairs of 2^20 coefficients: 4096 sampled coefficients (64 per
  pair) exact against the schoolbook sum; C(t) = A(t) B(t) mod 2^61 - 1 at two
  points for every pair (covers every coefficient).
* 32768 real signals x 3072 samples convolved with one 1025-tap filter: 16
  sampled rows against the direct sum.
* 16384 x 3000 (mixed radix) and 16384 x 3001 (Bluestein): 6 sampled rows
  against the direct DFT; the inverse round trip for every row.
* 32768 real rows x 8192: 16 sampled half spectra against the oracle; C2R
  round trip for every row.
* 4 volumes of 128 x 256 x 256: one volume against the oracle's separable
  3D transform; the inverse round trip for all four.

All floating-point bounds are the relative-L2 tolerance 1e-5 * log2(N).
"""
import multiprocessing as mp
import os
import tempfile
import threading

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL32 = 1e-5


@pytest.fixture(scope="module")
def fg(fg_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fg_lib


def rel_rows(y, ref):
    y = np.asarray(y, np.complex128).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.complex128).reshape(ref.shape[0], -1)
    return np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)


def _bins_worker(args):
    path, ks = args
    x = np.load(path, mmap_mode="r")
    return oracle.dft_bins(np.asarray(x), ks)


def test_c2_batched_4096(fg):
    c = workloads.CONFIGS["c2"]
    n, batch = c["n"], c["batch"]
    x = workloads.config_input("c2")
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty_like(xd)
    zd = torch.empty_like(xd)
    pf = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_C2C_F32)
    pi = fg.Plan(n, batch, 1, fg.FFT_INVERSE, fg.FFT_C2C_F32)
    pf.exec(xd, yd)
    pi.exec(yd, zd)
    torch.cuda.synchronize()
    idx = np.unique(workloads.sample_indices(48, batch, 21))
    y = yd[torch.from_numpy(idx).cuda()].cpu().numpy()
    ref = oracle.fft(x[idx].astype(np.complex128))
    assert rel_rows(y, ref).max() <= TOL32 * 12
    z = zd.cpu().numpy()
    assert rel_rows(z, x).max() <= 2 * TOL32 * 12
    assert fg.fft_device_status(int(torch.cuda.current_stream().cuda_stream)) == 0
    pf.close()
    pi.close()


def test_c3_single_2e26(fg):
    c = workloads.CONFIGS["c3"]
    n = c["n"]
    x = workloads.config_input("c3")[0]
    x64 = x.astype(np.complex128)
    # The oracle's recursive Cooley-Tukey of the whole vector (about half a
    # minute of one host core; the C call releases the GIL) runs while the
    # GPU transforms.
    full = {}
    worker = threading.Thread(target=lambda: full.setdefault("X", oracle.fft(x64)))
    worker.start()
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty_like(xd)
    zd = torch.empty_like(xd)
    pf = fg.Plan(n, 1, 1, fg.FFT_FORWARD, fg.FFT_C2C_F32)
    pi = fg.Plan(n, 1, 1, fg.FFT_INVERSE, fg.FFT_C2C_F32)
    pf.exec(xd, yd)
    pi.exec(yd, zd)
    torch.cuda.synchronize()
    y = yd.cpu().numpy().astype(np.complex128)
    z = zd.cpu().numpy().astype(np.complex128)
    # The 16 tone bins also against the direct DFT of those bins (an
    # independent oracle path), spread over spawned workers.
    bins, _, _ = workloads.tone_params(n, c["seed"])
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "x.npy")
        np.save(path, x64)
        chunks = [(path, bins[i::8]) for i in range(8)]
        with mp.get_context("spawn").Pool(8) as pool:
            parts = pool.map(_bins_worker, chunks)
    tone_ref = np.empty(bins.size, np.complex128)
    for i in range(8):
        tone_ref[i::8] = parts[i]
    worker.join()
    ref = full["X"]
    tol = TOL32 * 26
    # The whole vector: relative L2 error of the transform.
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) <= tol
    # Tone bins (magnitude N): relative error of each, against both oracle paths.
    assert np.max(np.abs(y[bins] - tone_ref) / np.abs(tone_ref)) <= tol
    assert np.max(np.abs(ref[bins] - tone_ref) / np.abs(tone_ref)) <= 1e-9
    assert np.all(np.abs(np.abs(tone_ref) - n) < 0.01 * n)
    # Parseval and the round trip over the whole vector.
    ex, eX = np.sum(np.abs(x64) ** 2), np.sum(np.abs(y) ** 2) / n
    assert abs(ex - eX) / ex <= tol
    assert np.linalg.norm(z - x64) / np.linalg.norm(x64) <= 2 * tol
    assert fg.fft_device_status(int(torch.cuda.current_stream().cuda_stream)) == 0
    pf.close()
    pi.close()


def test_c4_2d_2048(fg):
    c = workloads.CONFIGS["c4"]
    n, batch = c["n"], c["batch"]
    x = workloads.config_input("c4")
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty_like(xd)
    zd = torch.empty_like(xd)
    pf = fg.Plan(n, batch, 2, fg.FFT_FORWARD, fg.FFT_C2C_F32)
    pi = fg.Plan(n, batch, 2, fg.FFT_INVERSE, fg.FFT_C2C_F32)
    pf.exec(xd, yd)
    pi.exec(yd, zd)
    torch.cuda.synchronize()
    for b in (0, batch - 1):
        y = yd[b].cpu().numpy()
        ref = oracle.fft2d(x[b].astype(np.complex128))
        assert rel_rows(y[None], ref[None]).max() <= TOL32 * 22
    z = zd.cpu().numpy()
    assert rel_rows(z, x).max() <= 2 * TOL32 * 22
    pf.close()
    pi.close()


def test_c5_polymul_64_pairs(fg):
    c = workloads.CONFIGS["c5"]
    n, batch = c["n"], c["batch"]
    a, b = workloads.config_input("c5")
    cd = fg.polymul_tensors(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    out = cd.cpu().numpy()
    nc = 2 * n - 1
    assert out.shape == (batch, nc)
    for p in range(batch):
        idx = workloads.sample_indices(64, nc, 1000 + p)
        assert np.array_equal(out[p][idx], oracle.polymul_schoolbook_at(a[p], b[p], idx)), p
        for t in workloads.sample_indices(2, oracle.MOD_P, 2000 + p):
            t = int(t)
            lhs = oracle.poly_eval_mod(out[p], t)
            rhs = oracle.poly_eval_mod(a[p], t) * oracle.poly_eval_mod(b[p], t) % oracle.MOD_P
            assert lhs == rhs, p


def test_conv1_real_signals(fg):
    # 32768 real fp32 signals x 3072 samples, one 1025-tap real filter: 16
    # sampled rows (including the last) against the direct sum.
    c = workloads.CONFIGS["conv1"]
    x, h = workloads.config_input("conv1")
    y = fg.convolve(torch.from_numpy(x).cuda(), torch.from_numpy(h).cuda())
    torch.cuda.synchronize()
    ny = c["n"] + c["nh"] - 1
    assert tuple(y.shape) == (c["batch"], ny)
    rows = np.unique(np.concatenate([workloads.sample_indices(15, c["batch"], 61),
                                     [c["batch"] - 1]]))
    got = y[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.complex128)
    ref = oracle.convolve(x[rows].astype(np.complex128), h.astype(np.complex128))
    err = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert err.max() <= TOL32 * 12


def _any_length_full(fg, name):
    c = workloads.CONFIGS[name]
    n, batch = c["n"], c["batch"]
    x = workloads.config_input(name)
    xd = torch.from_numpy(x).cuda()
    yd, zd = torch.empty_like(xd), torch.empty_like(xd)
    pf = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_C2C_F32)
    pi = fg.Plan(n, batch, 1, fg.FFT_INVERSE, fg.FFT_C2C_F32)
    pf.exec(xd, yd)
    pi.exec(yd, zd)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([workloads.sample_indices(5, batch, 71), [batch - 1]]))
    y = yd[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref = np.stack([oracle.dft(x[r].astype(np.complex128)) for r in rows])
    tol = TOL32 * int(np.log2(n))
    assert rel_rows(y, ref).max() <= tol
    assert rel_rows(zd.cpu().numpy(), x).max() <= 2 * tol
    pf.close()
    pi.close()


def test_any1_mixed_radix_3000(fg):
    # 16384 x 3000 fp32 (mixed radix): 6 sampled rows (with the last) against
    # the direct DFT; the inverse returns every row.
    _any_length_full(fg, "any1")


def test_any2_bluestein_3001(fg):
    # 16384 x 3001 fp32 (prime: Bluestein, convolution length 8192).
    _any_length_full(fg, "any2")


def test_real1_r2c_c2r(fg):
    # 32768 real rows x 8192: 16 sampled half spectra (with the last row)
    # against the oracle; the C2R of the GPU spectra returns every row.
    c = workloads.CONFIGS["real1"]
    n, batch = c["n"], c["batch"]
    x = workloads.config_input("real1")
    xd = torch.from_numpy(x).cuda()
    pf = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_REAL_F32)
    pi = fg.Plan(n, batch, 1, fg.FFT_INVERSE, fg.FFT_REAL_F32)
    Xd = pf.exec(xd)
    zd = pi.exec(Xd)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([workloads.sample_indices(15, batch, 81), [batch - 1]]))
    X = Xd[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref = oracle.rfft(x[rows].astype(np.float64))
    assert rel_rows(X, ref).max() <= TOL32 * 13
    z = zd.cpu().numpy()
    err = np.linalg.norm(z - x, axis=1) / np.linalg.norm(x, axis=1)
    assert err.max() <= 2 * TOL32 * 13
    pf.close()
    pi.close()


def test_nd1_3d_volumes(fg):
    # 4 volumes of 128 x 256 x 256 fp32: volume 3 against the oracle's
    # separable transform; the inverse round trip for all four.
    c = workloads.CONFIGS["nd1"]
    shape, batch = tuple(c["shape"]), c["batch"]
    x = workloads.config_input("nd1")
    xd = torch.from_numpy(x).cuda()
    yd, zd = torch.empty_like(xd), torch.empty_like(xd)
    pf = fg.Plan(0, batch, direction=fg.FFT_FORWARD, dtype=fg.FFT_C2C_F32, shape=shape)
    pi = fg.Plan(0, batch, direction=fg.FFT_INVERSE, dtype=fg.FFT_C2C_F32, shape=shape)
    pf.exec(xd, yd)
    pi.exec(yd, zd)
    torch.cuda.synchronize()
    y3 = yd[3].cpu().numpy().reshape(1, -1)
    ref = oracle.fftn(x[3].astype(np.complex128), 3).reshape(1, -1)
    assert rel_rows(y3, ref).max() <= TOL32 * 23
    assert rel_rows(zd.cpu().numpy().reshape(batch, -1), x.reshape(batch, -1)).max() <= 2 * TOL32 * 23
    pf.close()
    pi.close()


@pytest.mark.parametrize("log_n,dtype", [(30, 0), (29, 1)])
def test_max_length_tones(fg, log_n, dtype):
    # The longest 1D plans (2^30 fp32 / 2^29 fp64 points, multi-pass, 8 GiB
    # per array): a sum of 8 unit tones at seeded integer bins has the exact
    # spectrum N at those bins and 0 elsewhere, so every output is checked;
    # the inverse returns the input.  (The input is formed on the device in
    # fp64 with every phase index reduced mod N in integers.)
    n = 1 << log_n
    bins, phases, _ = workloads.tone_params(n, 91 + log_n, ntones=8)
    dev = torch.device("cuda")
    idx = torch.arange(n, dtype=torch.int64, device=dev)
    re = torch.zeros(n, dtype=torch.float64, device=dev)
    im = torch.zeros(n, dtype=torch.float64, device=dev)
    for f, ph in zip(bins.tolist(), phases.tolist()):
        ang = (idx * f).remainder_(n).to(torch.float64).mul_(2 * np.pi / n).add_(2 * np.pi * ph)
        re += torch.cos(ang)
        im += torch.sin(ang)
        del ang
    del idx
    x = torch.complex(re.float(), im.float()) if dtype == 0 else torch.complex(re, im)
    del re, im
    y = torch.empty_like(x)
    pf = fg.Plan(n, 1, 1, fg.FFT_FORWARD, dtype)
    assert pf.num_kernels >= 3
    pf.exec(x, y)
    torch.cuda.synchronize()
    tol = (TOL32 if dtype == 0 else 1e-13) * log_n
    kb = torch.from_numpy(bins).to(dev)
    expect = torch.from_numpy(np.exp(2j * np.pi * phases).astype(np.complex128) * n).to(dev)
    at_tones = y[kb].clone()
    assert (at_tones.to(torch.complex128) - expect).abs().max().item() / n <= tol
    y[kb] = 0
    assert y.abs().max().item() / n <= tol
    y[kb] = at_tones
    pi = fg.Plan(n, 1, 1, fg.FFT_INVERSE, dtype)
    pi.exec(y, y)
    torch.cuda.synchronize()
    err = torch.linalg.vector_norm(y - x).item() / torch.linalg.vector_norm(x).item()
    assert err <= 2 * tol
    assert fg.fft_device_status(int(torch.cuda.current_stream().cuda_stream)) == 0
    pf.close()
    pi.close()
