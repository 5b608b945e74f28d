"""GPU parity: every transform the library runs, through the C ABI, against
the fp64 CPU oracle on the same seeded inputs.

Tolerances (relative L2 error per transform, maximum over the batch):
fp32 <= 1e-5 * log2(N), fp64 <= 1e-13 * log2(N), with N the number of
points of one transform (N*N for 2D).  Integer polynomial products are
compared bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32, F64 = 0, 1
TOL = {F32: 1e-5, F64: 1e-13}
NP = {F32: np.complex64, F64: np.complex128}


@pytest.fixture(scope="module")
def fg(fg_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fg_lib


def stream():
    return int(torch.cuda.current_stream().cuda_stream)


def rel_rows(y, ref):
    y = np.asarray(y, np.complex128).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.complex128).reshape(ref.shape[0], -1)
    num = np.linalg.norm(y - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    den[den == 0] = 1
    return num / den


def tol(dtype, npoints):
    return TOL[dtype] * max(1, int(np.log2(npoints)))


def run_plan(fg, x, n, batch, dims, direction, dtype, inplace=False):
    p = fg.Plan(n, batch, dims, direction, dtype)
    d = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = d if inplace else torch.empty_like(d)
    p.exec(d, out)
    torch.cuda.synchronize()
    y = out.cpu().numpy()
    p.close()
    return y


# --- batched 1D, on chip -------------------------------------------------------

@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("logn", list(range(0, 15)))
def test_rows_forward_inverse(fg, dtype, logn):
    if dtype == F64 and logn > 13:
        pytest.skip("fp64 on-chip limit is 2^13")
    n = 1 << logn
    batch = 5 if n >= 256 else 37   # ragged against the per-block transform count
    x = workloads.normal_complex((batch, n), 1000 + logn, NP[dtype])
    x64 = x.astype(np.complex128)
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype)
    ref = oracle.fft(x64)
    assert rel_rows(y, ref).max() <= tol(dtype, n)
    if n <= 1024:
        assert rel_rows(y[:2], np.stack([oracle.dft(r) for r in x64[:2]])).max() <= tol(dtype, n)
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, dtype)
    refi = oracle.ifft(y.astype(np.complex128))
    assert rel_rows(z, refi).max() <= tol(dtype, n)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_rows_in_place(fg, dtype):
    n, batch = 4096, 9
    x = workloads.uniform_complex((batch, n), 7, NP[dtype])
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype, inplace=True)
    assert rel_rows(y, oracle.fft(x.astype(np.complex128))).max() <= tol(dtype, n)


def test_rows_closed_forms(fg):
    n = 2048
    x = np.zeros((3, n), np.complex64)
    x[0, 0] = 1                                    # delta -> all ones
    x[1, :] = 0.5 - 0.25j                          # constant -> N c at bin 0
    f = 77                                         # single integer tone -> N at bin f
    x[2] = np.exp(2j * np.pi * ((f * np.arange(n)) % n) / n)
    y = run_plan(fg, x, n, 3, 1, fg.FFT_FORWARD, F32)
    assert np.max(np.abs(y[0] - 1)) < 1e-6
    assert abs(y[1, 0] - n * (0.5 - 0.25j)) < 1e-3 and np.max(np.abs(y[1, 1:])) < 1e-3
    e = np.zeros(n)
    e[f] = n
    assert np.max(np.abs(y[2] - e)) < 5e-3


# --- long 1D: multi-pass -------------------------------------------------------

@pytest.mark.parametrize("dtype,logn", [(F32, 15), (F32, 16), (F32, 18), (F32, 19), (F32, 20),
                                        (F64, 14), (F64, 15), (F64, 17), (F64, 19)])
def test_multipass_forward_inverse(fg, dtype, logn):
    n = 1 << logn
    batch = 2
    x = workloads.normal_complex((batch, n), 2000 + logn, NP[dtype])
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype)
    assert rel_rows(y, oracle.fft(x.astype(np.complex128))).max() <= tol(dtype, n)
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, dtype, inplace=True)
    assert rel_rows(z, oracle.ifft(y.astype(np.complex128))).max() <= tol(dtype, n)


@pytest.mark.parametrize("passlog", [5, 7, 9, 13])
def test_multipass_factorisations(fg, opt, passlog):
    # The same 2^18 transform split into 2, 3 or 4 passes.
    opt("PASS_LOG", passlog)
    n = 1 << 18
    x = workloads.uniform_complex((1, n), 31, np.complex64)
    y = run_plan(fg, x, n, 1, 1, fg.FFT_FORWARD, F32)
    assert rel_rows(y, oracle.fft(x.astype(np.complex128))).max() <= tol(F32, n)


@pytest.mark.parametrize("dims,dtype,logn", [(1, F32, 18), (1, F32, 22), (1, F64, 17),
                                              (2, F32, 11), (2, F64, 9)])
def test_lsu_pass_kernel(fg, opt, dims, dtype, logn):
    # The pass kernel with plain loads/stores (what runs when the TMA path
    # does not apply) on shapes that normally take the TMA path.
    opt("NO_TMA", 1)
    n = 1 << logn
    shape = (1, n) if dims == 1 else (1, n, n)
    x = workloads.normal_complex(shape, 5000 + logn, NP[dtype])
    y = run_plan(fg, x, n, 1, dims, fg.FFT_FORWARD, dtype)
    ref = oracle.fft(x.astype(np.complex128)) if dims == 1 else np.fft.fft2(x.astype(np.complex128))
    npts = n if dims == 1 else n * n
    assert rel_rows(y, ref).max() <= tol(dtype, npts)


# 512-point transforms with the warp-shuffle exchange (FFT_OPT_ROWS_SHFL): one
# warp per transform, four register/lane bit swaps by __shfl_xor_sync and a
# final 2-point butterfly across lane pairs; ragged batches against the
# oracle, forward and inverse, in place and out of place.
@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("batch", [1, 7, 8, 61])
def test_rows_warp_shuffle_512(fg, opt, dtype, batch):
    opt("ROWS_SHFL", 1)
    n = 512
    x = workloads.normal_complex((batch, n), 3900 + batch, NP[dtype])
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype)
    assert rel_rows(y, oracle.fft(x.astype(np.complex128))).max() <= tol(dtype, n)
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, dtype, inplace=True)
    assert rel_rows(z, oracle.ifft(y.astype(np.complex128))).max() <= tol(dtype, n)


# 512-point fp32 HBM passes with the warp-shuffle exchange (FFT_OPT_PASS_SHFL):
# one warp per column, tiles moved with the TMA's 64-byte swizzle.  Splits put
# the 512-point pass first (m = 1, linear bulk stores), in the middle and last
# (twiddled, TMA stores), with blocks of m down to one tile (m = 8); the 2D
# shapes run it as the column pass (folded and not), in and out of place.
@pytest.mark.parametrize("logn,split,batch", [
    (18, "9,9", 2), (21, "3,9,9", 1), (13, "4,9", 3), (12, "3,9", 2), (17, "9,8", 1),
    (22, "9,9,4", 1)])
def test_pass_warp_shuffle(fg, opt, logn, split, batch):
    opt("PASS_SPLIT", split)
    opt("PASS_SHFL", 1)
    n = 1 << logn
    x = workloads.normal_complex((batch, n), 6400 + logn, np.complex64)
    ref = oracle.fft(x.astype(np.complex128))
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, F32)
    assert rel_rows(y, ref).max() <= tol(F32, n)
    y2 = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, F32, inplace=True)
    assert rel_rows(y2, ref).max() <= tol(F32, n)
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, F32)
    assert rel_rows(z, oracle.ifft(y.astype(np.complex128))).max() <= tol(F32, n)
    assert fg.fft_device_status(stream()) == 0


@pytest.mark.parametrize("shape,batch", [((2048, 2048), 2), ((512, 512), 3), ((512, 256), 2),
                                         ((1024, 64), 2)])
def test_pass_warp_shuffle_2d(fg, opt, shape, batch):
    opt("PASS_SHFL", 1)
    x = workloads.normal_complex((batch,) + shape, 6500 + sum(shape), np.complex64)
    npts = int(np.prod(shape))
    p = fg.Plan(0, batch, direction=fg.FFT_FORWARD, dtype=F32, shape=shape)
    pi = fg.Plan(0, batch, direction=fg.FFT_INVERSE, dtype=F32, shape=shape)
    xd = torch.from_numpy(x).cuda()
    yd, zd = torch.empty_like(xd), torch.empty_like(xd)
    p.exec(xd, yd)
    pi.exec(yd, zd)
    torch.cuda.synchronize()
    ref = oracle.fftn(x.astype(np.complex128), 2)
    assert rel_rows(yd.cpu().numpy(), ref).max() <= tol(F32, npts)
    assert rel_rows(zd.cpu().numpy(), x).max() <= 2 * tol(F32, npts)
    p.exec(xd, xd)
    torch.cuda.synchronize()
    assert rel_rows(xd.cpu().numpy(), ref).max() <= tol(F32, npts)
    assert fg.fft_device_status(stream()) == 0
    p.close()
    pi.close()


# --- passes whose on-chip length (2^11 .. 2^13) is split over a cluster --------

@pytest.mark.parametrize("dtype,logn,split,batch", [
    (F32, 22, "11,11", 1),   # clusters of 2 in both passes
    (F32, 20, "13,7", 2),    # clusters of 8 in the first pass (linear stores)
    (F32, 20, "7,13", 2),    # clusters of 8 in the last pass (twiddled, TMA stores)
    (F32, 24, "12,12", 1),   # clusters of 4
    (F32, 17, "4,13", 3),    # last pass with m = 16 (four tiles per block of m)
    (F32, 15, "13,2", 2),    # first pass with 4 columns: one tile per transform
    (F32, 21, "7,12,2", 1),  # a middle pass
    (F64, 21, "11,10", 1),
    (F64, 20, "8,12", 2),
])
def test_cluster_passes(fg, opt, dtype, logn, split, batch):
    opt("PASS_SPLIT", split)
    opt("CLUSTER_LOG_MIN", 11)  # clusters of 2 as well
    n = 1 << logn
    x = workloads.normal_complex((batch, n), 6000 + logn, NP[dtype])
    ref = oracle.fft(x.astype(np.complex128))
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype)
    assert rel_rows(y, ref).max() <= tol(dtype, n)
    y2 = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype, inplace=True)
    assert rel_rows(y2, ref).max() <= tol(dtype, n)
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, dtype)
    assert rel_rows(z, oracle.ifft(y.astype(np.complex128))).max() <= tol(dtype, n)
    assert fg.fft_device_status(stream()) == 0


@pytest.mark.parametrize("split", ["13,11", "11,13", "12,12", "8,8,8"])
def test_cluster_pass_splits_2e24(fg, opt, split):
    # One 2^24 transform split into cluster passes of 2^11 .. 2^13 points
    # (and, for comparison, into single-block passes), against the oracle at
    # every bin, forward and inverse.
    opt("PASS_SPLIT", split)
    opt("CLUSTER_LOG_MIN", 11)
    n = 1 << 24
    x = workloads.normal_complex((1, n), 6100, np.complex64)
    y = run_plan(fg, x, n, 1, 1, fg.FFT_FORWARD, F32)
    assert rel_rows(y, oracle.fft(x.astype(np.complex128))).max() <= tol(F32, n)
    z = run_plan(fg, y, n, 1, 1, fg.FFT_INVERSE, F32, inplace=True)
    assert rel_rows(z, x.astype(np.complex128)).max() <= 2 * tol(F32, n)


def test_cluster_pass_disabled_fallback(fg, opt):
    # FFT_OPT_NO_CLUSTER: the same split runs on the single-block kernels.
    opt("PASS_SPLIT", "12,10")
    opt("NO_CLUSTER", 1)
    n = 1 << 22
    x = workloads.uniform_complex((1, n), 6200, np.complex64)
    y = run_plan(fg, x, n, 1, 1, fg.FFT_FORWARD, F32)
    assert rel_rows(y, oracle.fft(x.astype(np.complex128))).max() <= tol(F32, n)


def test_device_status_clear_after_transforms(fg):
    # No bounded in-kernel wait ran out during the transforms above.
    assert fg.fft_device_status(stream()) == 0


# --- 2D -----------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("logn", [0, 1, 2, 4, 5, 7, 8, 9])
def test_2d_forward_inverse(fg, dtype, logn):
    n = 1 << logn
    batch = 3
    x = workloads.normal_complex((batch, n, n), 3000 + logn, NP[dtype])
    y = run_plan(fg, x, n, batch, 2, fg.FFT_FORWARD, dtype)
    ref = oracle.fft2d(x.astype(np.complex128))
    assert rel_rows(y, ref).max() <= tol(dtype, n * n)
    z = run_plan(fg, y, n, batch, 2, fg.FFT_INVERSE, dtype)
    assert rel_rows(z, oracle.fft2d(y.astype(np.complex128), +1)).max() <= tol(dtype, n * n)


@pytest.mark.parametrize("dtype,logn", [(F32, 11), (F32, 12), (F32, 13), (F64, 11), (F64, 12)])
def test_2d_large_sides(fg, dtype, logn):
    n = 1 << logn
    x = workloads.uniform_complex((1, n, n), 3100 + logn, NP[dtype])
    y = run_plan(fg, x, n, 1, 2, fg.FFT_FORWARD, dtype)
    # separable check against numpy's 2D FFT computed in fp64 (independent)
    ref = np.fft.fft2(x.astype(np.complex128))
    assert rel_rows(y, ref).max() <= tol(dtype, n * n)
    if logn <= 11:
        assert rel_rows(y, oracle.fft2d(x.astype(np.complex128))).max() <= tol(dtype, n * n)


@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("shape", [(2, 8), (64, 32), (16, 1024), (1024, 16), (4, 8, 16),
                                   (32, 16, 64), (2, 2, 2), (1, 16, 16), (128, 1, 4), (8, 4, 1),
                                   (2048, 8), (4096, 4), (8192, 2), (2, 4096, 4)])
def test_nd_forward_inverse(fg, dtype, shape):
    batch = 3
    x = workloads.normal_complex((batch,) + shape, 3500 + sum(shape), NP[dtype])
    npts = int(np.prod(shape))
    p = fg.Plan(0, batch, direction=fg.FFT_FORWARD, dtype=dtype, shape=shape)
    pi = fg.Plan(0, batch, direction=fg.FFT_INVERSE, dtype=dtype, shape=shape)
    d = torch.from_numpy(x).cuda()
    y = p.exec(d)
    z = pi.exec(y)
    torch.cuda.synchronize()
    ref = oracle.fftn(x.astype(np.complex128), len(shape))
    assert rel_rows(y.cpu().numpy(), ref).max() <= tol(dtype, npts)
    assert rel_rows(z.cpu().numpy(), x).max() <= 2 * tol(dtype, npts)
    p.close()
    pi.close()


# Columns of 1024 points or more, out of place: the row pass also takes the
# first radix-R stage of the column transform (R = H / 512 up to 2048
# points, R = 4 or 2 for 4096 and 8192) and the column pass transforms
# columns H / R long, R W apart.  In place the plan keeps rows plus a full
# column pass; both schedules are checked against the oracle.
@pytest.mark.parametrize("dtype,shape,batch", [
    (F32, (1024, 256), 3), (F32, (2048, 256), 2), (F64, (2048, 256), 2), (F32, (4096, 256), 1),
    (F64, (4096, 256), 1), (F32, (2048, 2048), 2), (F32, (4096, 1024), 1), (F32, (1024, 4096), 1),
    (F64, (1024, 2048), 1), (F32, (2, 1024, 256), 2), (F64, (4, 2048, 512), 1),
    (F32, (4096, 4096), 1), (F32, (8192, 1024), 1), (F32, (8192, 256), 2), (F64, (8192, 512), 1),
    (F32, (2, 4096, 256), 1)])
def test_nd_folded_column_radix(fg, dtype, shape, batch):
    x = workloads.normal_complex((batch,) + shape, 3600 + sum(shape), NP[dtype])
    npts = int(np.prod(shape))
    p = fg.Plan(0, batch, direction=fg.FFT_FORWARD, dtype=dtype, shape=shape)
    pi = fg.Plan(0, batch, direction=fg.FFT_INVERSE, dtype=dtype, shape=shape)
    assert p.num_kernels == len(shape)
    xd = torch.from_numpy(x).cuda()
    yd, zd = torch.empty_like(xd), torch.empty_like(xd)
    p.exec(xd, yd)
    pi.exec(yd, zd)
    torch.cuda.synchronize()
    ref = oracle.fftn(x.astype(np.complex128), len(shape))
    assert rel_rows(yd.cpu().numpy(), ref).max() <= tol(dtype, npts)
    assert rel_rows(zd.cpu().numpy(), x).max() <= 2 * tol(dtype, npts)
    assert np.array_equal(xd.cpu().numpy(), x)          # input untouched
    p.exec(xd, xd)                                      # in place: rows + column pass
    torch.cuda.synchronize()
    assert rel_rows(xd.cpu().numpy(), ref).max() <= tol(dtype, npts)
    p.close()
    pi.close()


@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("shape", [(8192, 2), (2048, 4), (4096, 8)])
def test_nd_columns_single_block(fg, opt, dtype, shape):
    # Long columns on the single-block pass kernels (FFT_OPT_NO_CLUSTER);
    # fp64 columns of 8192 compute their stage twiddles (no shared table).
    opt("NO_CLUSTER", 1)
    x = workloads.normal_complex((2,) + shape, 3550 + sum(shape), NP[dtype])
    p = fg.Plan(0, 2, direction=fg.FFT_FORWARD, dtype=dtype, shape=shape)
    y = p.exec(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    ref = oracle.fftn(x.astype(np.complex128), len(shape))
    assert rel_rows(y.cpu().numpy(), ref).max() <= tol(dtype, int(np.prod(shape)))
    p.close()


def test_nd_large_3d(fg):
    shape = (256, 512, 64)        # 8 Mi points: rows of 64, columns of 512 and 256
    x = workloads.uniform_complex((1,) + shape, 3600, np.complex64)
    y = fg.fftn(torch.from_numpy(x).cuda(), 3)
    torch.cuda.synchronize()
    ref = oracle.fftn(x.astype(np.complex128), 3)
    assert rel_rows(y.cpu().numpy(), ref).max() <= tol(F32, int(np.prod(shape)))


# Every axis as on-chip rows with transposed stores: the default when every
# side is 128 or 256, forced here (FFT_OPT_ND_ROWS_T = 1) on other sides
# too; out of place and in place (rank 3 in place ends with a copy).
@pytest.mark.parametrize("dtype,shape,force", [
    (F32, (128, 256), False), (F32, (256, 256), False), (F32, (128, 128, 256), False),
    (F32, (64, 32), True), (F32, (16, 1024), True), (F32, (4096, 16), True),
    (F32, (32, 16, 64), True), (F64, (256, 128), False), (F64, (64, 4096), True), (F64, (64, 8192), True),
    (F64, (16, 32, 64), True)])
def test_nd_rows_transposed(fg, opt, dtype, shape, force):
    if force:
        opt("ND_ROWS_T", 1)
    batch = 3
    x = workloads.normal_complex((batch,) + shape, 3700 + sum(shape), NP[dtype])
    p = fg.Plan(0, batch, direction=fg.FFT_FORWARD, dtype=dtype, shape=shape)
    pi = fg.Plan(0, batch, direction=fg.FFT_INVERSE, dtype=dtype, shape=shape)
    assert p.num_kernels == len(shape)
    # Sides beyond the transposed-store limit (2^12) keep the column passes.
    assert (p.workspace_bytes > 0) == (max(shape) <= 4096)
    d = torch.from_numpy(x).cuda()
    y = p.exec(d)
    z = pi.exec(y)
    torch.cuda.synchronize()
    npts = int(np.prod(shape))
    ref = oracle.fftn(x.astype(np.complex128), len(shape))
    assert rel_rows(y.cpu().numpy(), ref).max() <= tol(dtype, npts)
    assert rel_rows(z.cpu().numpy(), x).max() <= 2 * tol(dtype, npts)
    p.exec(d, d)
    torch.cuda.synchronize()
    assert rel_rows(d.cpu().numpy(), ref).max() <= tol(dtype, npts)
    p.close()
    pi.close()


def test_nd_rejects(fg):
    with pytest.raises(fg.FFTError):
        fg.Plan(0, 1, shape=(6, 0))                 # empty side
    with pytest.raises(fg.FFTError):
        fg.Plan(0, 1, shape=(2, 1 << 31))           # side beyond 2^30
    with pytest.raises(fg.FFTError):
        fg.fft_plan_create_nd(4, (2, 2, 2, 2), 1, -1, 0)


# Sides that are not powers of two, or beyond one kernel per axis: the
# contiguous axis as a 1D plan of any length, the others as power-of-two
# column passes or between two transposes.
@pytest.mark.parametrize("dtype,shape,batch", [
    (F32, (6, 8), 3), (F32, (100, 64), 2), (F32, (30, 50), 2), (F32, (3, 5, 7), 3),
    (F32, (12, 16, 20), 2), (F32, (7, 1, 9), 2), (F32, (1, 100), 3), (F32, (64, 3000), 2),
    (F32, (2, 2, 1 << 15), 2), (F32, (1 << 15, 4), 2), (F32, (1009, 6), 2),
    (F64, (6, 8), 3), (F64, (30, 50), 2), (F64, (12, 16, 20), 2), (F64, (1 << 14, 4), 1)])
def test_nd_any_sides(fg, dtype, shape, batch):
    x = workloads.normal_complex((batch,) + shape, 5600 + sum(shape), NP[dtype])
    p = fg.Plan(0, batch, direction=fg.FFT_FORWARD, dtype=dtype, shape=shape)
    pi = fg.Plan(0, batch, direction=fg.FFT_INVERSE, dtype=dtype, shape=shape)
    xd = torch.from_numpy(x).cuda()
    yd, zd = torch.empty_like(xd), torch.empty_like(xd)
    p.exec(xd, yd)
    pi.exec(yd, zd)
    torch.cuda.synchronize()
    npts = int(np.prod(shape))
    t = tol(dtype, npts)
    ref = oracle.fftn(x.astype(np.complex128), len(shape))
    assert rel_rows(yd.cpu().numpy(), ref).max() <= t
    assert rel_rows(zd.cpu().numpy(), x).max() <= 2 * t
    # in place
    p.exec(xd, xd)
    torch.cuda.synchronize()
    assert rel_rows(xd.cpu().numpy(), ref).max() <= t
    p.close()
    pi.close()


# --- lengths that are not powers of two ---------------------------------------

@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("n", [3, 5, 6, 12, 17, 33, 63])
def test_direct_dft_short_lengths(fg, dtype, n):
    batch = 37
    x = workloads.normal_complex((batch, n), 5200 + n, NP[dtype])
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype)
    ref = np.stack([oracle.dft(r) for r in x.astype(np.complex128)])
    assert rel_rows(y, ref).max() <= tol(dtype, n)
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, dtype, inplace=True)
    assert rel_rows(z, x).max() <= 2 * tol(dtype, n)


@pytest.mark.parametrize("dtype,n", [(F32, 67), (F32, 134), (F32, 1009), (F32, 3001), (F32, 8191),
                                     (F64, 67), (F64, 1009), (F64, 4091),
                                     (F32, 10007), (F64, 5003), (F64, 9999)])
def test_bluestein(fg, dtype, n):
    # Lengths with a prime factor above 13.  n <= 8191 fp32 / 4096 fp64 fuse
    # the whole convolution on chip; the rest take the multi-pass path.
    batch = 3
    x = workloads.normal_complex((batch, n), 5300 + n, NP[dtype])
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype)
    ref = np.stack([oracle.dft(r) for r in x.astype(np.complex128)])
    t = tol(dtype, n)
    assert rel_rows(y, ref).max() <= t
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, dtype, inplace=True)
    assert rel_rows(z, x).max() <= 2 * t


# Lengths whose prime factors are 2, 3, 5, 7, 11, 13 (above the direct-DFT
# range): mixed-radix stages on chip, one kernel.
@pytest.mark.parametrize("dtype,n", [(F32, 72), (F32, 96), (F32, 100), (F32, 120), (F32, 210),
                                     (F32, 243), (F32, 343), (F32, 625), (F32, 1000), (F32, 3000),
                                     (F32, 5040), (F32, 11025), (F32, 12288),
                                     (F32, 65), (F32, 121), (F32, 143), (F32, 169), (F32, 1001),
                                     (F32, 1331), (F32, 2197), (F32, 6656), (F32, 11264),
                                     (F64, 72), (F64, 210), (F64, 1000), (F64, 3000), (F64, 6144),
                                     (F64, 143), (F64, 4004), (F64, 2197)])
def test_mixed_radix(fg, dtype, n):
    batch = 3 if n > 2048 else 37   # ragged against the transforms per block
    x = workloads.normal_complex((batch, n), 5400 + n, NP[dtype])
    p = fg.Plan(n, batch, 1, fg.FFT_FORWARD, dtype)
    assert p.num_kernels == 1
    p.close()
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype)
    rows = range(batch) if n <= 3000 else range(2)
    ref = np.stack([oracle.dft(x[r].astype(np.complex128)) for r in rows])
    assert rel_rows(y[list(rows)], ref).max() <= tol(dtype, n)
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, dtype, inplace=True)
    assert rel_rows(z, x).max() <= 2 * tol(dtype, n)
    refi = np.stack([oracle.dft(y[r].astype(np.complex128), +1) for r in rows])
    assert rel_rows(z[list(rows)], refi).max() <= tol(dtype, n)


# Smooth lengths beyond one block: four-step N = N1 N2 with both factors on
# chip (transpose, N1-point transforms, twiddled transpose, N2-point
# transforms, transpose); 16 sampled bins of two rows against the direct sum,
# Parseval, the inverse round trip, and the in-place form.
@pytest.mark.parametrize("dtype,n", [(F32, 12800), (F32, 100000), (F32, 59049), (F32, 78125),
                                     (F32, 53760), (F32, 15488), (F32, 28561), (F64, 24576),
                                     (F64, 10000), (F64, 8788)])
def test_four_step_smooth(fg, dtype, n):
    batch = 3
    x = workloads.normal_complex((batch, n), 5500 + n % 997, NP[dtype])
    p = fg.Plan(n, batch, 1, fg.FFT_FORWARD, dtype)
    assert p.num_kernels >= 5 and p.workspace_bytes > 0
    p.close()
    y = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype)
    t = tol(dtype, n)
    ks = np.unique(np.concatenate([workloads.sample_indices(14, n, 5501), [0, n - 1]]))
    for r in (0, batch - 1):
        x64 = x[r].astype(np.complex128)
        ref = oracle.dft_bins(x64, ks)
        rms = np.linalg.norm(y[r]) / np.sqrt(n)
        assert np.linalg.norm(y[r][ks] - ref) / (np.sqrt(ks.size) * rms) <= t
        assert abs(np.sum(np.abs(x64) ** 2) - np.sum(np.abs(y[r].astype(np.complex128)) ** 2) / n) \
            <= t * np.sum(np.abs(x64) ** 2)
    z = run_plan(fg, y, n, batch, 1, fg.FFT_INVERSE, dtype, inplace=True)
    assert rel_rows(z, x).max() <= 2 * t
    w = run_plan(fg, x, n, batch, 1, fg.FFT_FORWARD, dtype, inplace=True)
    assert rel_rows(w, y).max() <= t


def test_bluestein_large_prime_sampled(fg):
    n = 1000003                     # prime; convolution length 2^21 (3 passes)
    x = workloads.normal_complex((1, n), 54, np.complex64)
    y = run_plan(fg, x, n, 1, 1, fg.FFT_FORWARD, F32)[0].astype(np.complex128)
    ks = workloads.sample_indices(12, n, 55)
    ref = oracle.dft_bins(x[0].astype(np.complex128), ks)
    rms = np.linalg.norm(y) / np.sqrt(n)
    assert np.linalg.norm(y[ks] - ref) / (np.sqrt(ks.size) * rms) <= tol(F32, n)
    x64 = x[0].astype(np.complex128)
    assert abs(np.sum(np.abs(x64) ** 2) - np.sum(np.abs(y) ** 2) / n) / np.sum(np.abs(x64) ** 2) \
        <= tol(F32, n)


def test_bluestein_in_host_chain(fg):
    n, batch = 1500, 6
    x = workloads.normal_complex((batch, n), 56, np.complex64)
    pf = fg.Plan(n, batch, 1, fg.FFT_FORWARD, F32)
    pi = fg.Plan(n, batch, 1, fg.FFT_INVERSE, F32)
    h_in = torch.from_numpy(x).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    da, db = torch.empty_like(h_in).cuda(), torch.empty_like(h_in).cuda()
    pf.chain_host([pi], h_in, h_out, da, db, 4)
    torch.cuda.synchronize()
    assert rel_rows(h_out.numpy(), x).max() <= 2 * tol(F32, n)
    assert pf.num_kernels == 1 and pf.workspace_bytes > 0
    pf.close()
    pi.close()


# --- polynomial multiplication ----------------------------------------------

@pytest.mark.parametrize("na,nb,batch", [(1, 1, 1), (1, 5, 2), (5, 7, 3), (16, 16, 4),
                                         (100, 1000, 2), (1000, 3000, 2), (4096, 4096, 3),
                                         (4097, 10, 1), (1 << 15, 1 << 15, 2)])
def test_polymul_exact(fg, na, nb, batch):
    g = workloads.generator(na * 7 + nb)
    a = g.integers(0, 10, size=(batch, na), dtype=np.int64)
    b = g.integers(0, 10, size=(batch, nb), dtype=np.int64)
    c = fg.polymul_tensors(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    c = c.cpu().numpy()
    for p in range(batch):
        if na * nb <= 1 << 24:
            assert np.array_equal(c[p], oracle.polymul_schoolbook(a[p], b[p]))
        else:
            idx = workloads.sample_indices(512, na + nb - 1, p)
            assert np.array_equal(c[p][idx], oracle.polymul_schoolbook_at(a[p], b[p], idx))
            assert np.array_equal(c[p], oracle.polymul_fft(a[p], b[p]))


def test_polymul_three_pass_forward(fg):
    # L = 2^23: the forward transform takes three passes (the inter-pass
    # twiddle tables serve a pass with L m < L), the inverse two.
    na = nb = 1 << 22
    g = workloads.generator(23)
    a = g.integers(0, 10, size=na, dtype=np.int64)
    b = g.integers(0, 10, size=nb, dtype=np.int64)
    c = fg.polymul_tensors(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    c = c.cpu().numpy()
    idx = workloads.sample_indices(48, na + nb - 1, 24)
    assert np.array_equal(c[idx], oracle.polymul_schoolbook_at(a, b, idx))
    for t in (3, 123456789):
        assert oracle.poly_eval_mod(c, t) == \
            oracle.poly_eval_mod(a, t) * oracle.poly_eval_mod(b, t) % oracle.MOD_P


def test_polymul_kernel_count(fg):
    assert fg.polymul_num_kernels(1 << 20, 1 << 20) == 7   # 3 tables, 2 + 2 passes (product fused)
    assert fg.polymul_num_kernels(0, 5) == 0


def test_polymul_signed_coefficients(fg):
    g = workloads.generator(5)
    a = g.integers(-1000, 1001, size=3000, dtype=np.int64)
    b = g.integers(-1000, 1001, size=2000, dtype=np.int64)
    c = fg.polymul_tensors(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().numpy(), oracle.polymul_schoolbook(a, b))


# --- the single butterfly pass ------------------------------------------------

@pytest.mark.parametrize("dtype", [F32, F64])
def test_radix2_pass_8_points(fg, dtype):
    s = workloads.p1_spectrum().astype(NP[dtype])
    d = torch.from_numpy(s).cuda()
    y = d
    for half in (1, 2, 4):
        out = torch.empty_like(d)
        assert fg.fft_debug_radix2_pass(d.data_ptr(), out.data_ptr(), 8, half, dtype,
                                        stream()) == 0
        torch.cuda.synchronize()
        ref = oracle.radix2_pass(s.astype(np.complex128), half)
        assert np.max(np.abs(out.cpu().numpy() - ref)) < (1e-6 if dtype == F32 else 1e-15)
    # bit-reversed input through half = 1, 2, 4 is the 8-point DFT
    y = torch.from_numpy(oracle.bit_reverse(s.astype(np.complex128)).astype(NP[dtype])).cuda()
    for half in (1, 2, 4):
        out = torch.empty_like(y)
        assert fg.fft_debug_radix2_pass(y.data_ptr(), out.data_ptr(), 8, half, dtype,
                                        stream()) == 0
        y = out
    torch.cuda.synchronize()
    assert rel_rows(y.cpu().numpy()[None], oracle.dft(s.astype(np.complex128))[None]).max() \
        <= tol(dtype, 8)


def test_radix2_pass_large(fg):
    n = 1 << 16
    x = workloads.normal_complex(n, 9, np.complex64)
    d = torch.from_numpy(x).cuda()
    for half in (1, 8, 1 << 15):
        out = torch.empty_like(d)
        assert fg.fft_debug_radix2_pass(d.data_ptr(), out.data_ptr(), n, half, F32, stream()) == 0
        torch.cuda.synchronize()
        ref = oracle.radix2_pass(x.astype(np.complex128), half)
        assert rel_rows(out.cpu().numpy()[None], ref[None]).max() < 1e-6


# --- host-staged pipeline --------------------------------------------------

@pytest.mark.parametrize("n,dims,batch,chunk", [(4096, 1, 10, 3), (1 << 16, 1, 5, 2),
                                                (64, 2, 7, 4), (512, 1, 4, 9)])
def test_exec_host_chain_matches_device_exec(fg, n, dims, batch, chunk):
    # Forward then inverse over host buffers in chunks equals the same two
    # plans run on device buffers (bit for bit: same kernels, same data).
    shape = (batch, n) if dims == 1 else (batch, n, n)
    x = workloads.normal_complex(shape, 60 + n, np.complex64)
    pf = fg.Plan(n, batch, dims, fg.FFT_FORWARD, F32)
    pi = fg.Plan(n, batch, dims, fg.FFT_INVERSE, F32)
    h_in = torch.from_numpy(x).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    da = torch.empty(shape, dtype=torch.complex64, device="cuda")
    db = torch.empty_like(da)
    pf.chain_host([pi], h_in, h_out, da, db, chunk)
    torch.cuda.synchronize()
    d = torch.from_numpy(x).cuda()
    y = pi.exec(pf.exec(d))
    torch.cuda.synchronize()
    assert np.array_equal(h_out.numpy(), y.cpu().numpy())
    # one plan: the forward result lands in host_out
    pf.chain_host([], h_in, h_out, da, db, chunk)
    torch.cuda.synchronize()
    assert np.array_equal(h_out.numpy(), pf.exec(d).cpu().numpy())
    pf.close()
    pi.close()


# --- error reporting on a GPU ------------------------------------------------

def test_bounded_wait_reports_timeout(fg):
    # A wait that runs out is reported through the device status word, the
    # word is cleared by reading it, and the context stays usable.
    assert fg.fft_device_status(stream()) == 0
    assert fg.fft_debug_wait_timeout(2000, stream()) == 0
    assert fg.fft_device_status(stream()) == fg.FFT_ERR_DEVICE_TIMEOUT
    assert fg.fft_device_status(stream()) == 0
    x = workloads.uniform_complex((2, 1024), 3, np.complex64)
    y = run_plan(fg, x, 1024, 2, 1, fg.FFT_FORWARD, F32)
    assert rel_rows(y, oracle.fft(x.astype(np.complex128))).max() <= tol(F32, 1024)
    assert fg.fft_debug_wait_timeout(0, stream()) == fg.FFT_ERR_INVALID_ARG


def test_cluster_pass_timeout_reported(fg):
    # One block of a cluster waits for a tile load that never completes: the
    # whole cluster leaves after the bounded wait, the status word says so,
    # and the next cluster pass on the context is correct.
    buf = torch.zeros(1 << 15, dtype=torch.complex64, device="cuda")
    assert fg.fft_debug_cluster_timeout(buf.data_ptr(), 2000, stream()) == 0
    assert fg.fft_device_status(stream()) == fg.FFT_ERR_DEVICE_TIMEOUT
    assert fg.fft_device_status(stream()) == 0
    x = workloads.normal_complex((1, 8192, 8), 6300, np.complex64)
    p = fg.Plan(0, 1, direction=fg.FFT_FORWARD, dtype=F32, shape=(8192, 8))
    y = p.exec(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert rel_rows(y.cpu().numpy(), oracle.fftn(x.astype(np.complex128), 2)).max() <= \
        tol(F32, 8192 * 8)
    p.close()
    assert fg.fft_device_status(stream()) == 0
    assert fg.fft_debug_cluster_timeout(buf.data_ptr(), 0, stream()) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_cluster_timeout(buf.data_ptr() + 8, 10, stream()) == fg.FFT_ERR_MISALIGNED


def test_misaligned_device_pointer(fg):
    p = fg.Plan(64, 1, 1, fg.FFT_FORWARD, F32)
    buf = torch.zeros(2 * 64 + 8, dtype=torch.complex64, device="cuda")
    assert fg.fft_exec(p.handle, buf.data_ptr() + 8, buf.data_ptr() + 1024, stream()) == \
        fg.FFT_ERR_MISALIGNED
    p.close()
