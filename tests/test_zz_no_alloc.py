"""polymul_noalloc: the polynomial product for callers that cannot allocate
device memory where they need it (a plug-in inside a host application that
owns the memory budget, a latency-critical loop).  Its scratch is a fixed
array inside the library, so every call must give the exact product -- the
oracle's schoolbook sum, and the same bits as the allocating entry point --
also on later calls that find an earlier call's data still in that array.
Kept in its own file, collected last."""
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


def _both(fg, a_h, b_h):
    """(polymul's product, polymul_noalloc's product) of the same inputs."""
    na, nb = a_h.size, b_h.size
    a = torch.from_numpy(a_h).cuda()
    b = torch.from_numpy(b_h).cuda()
    c_ref = torch.empty(na + nb - 1, dtype=torch.int64, device="cuda")
    # Filled with a value no product here can take, so an output the call
    # leaves unwritten shows.
    c_new = torch.full((na + nb - 1,), -(1 << 62), dtype=torch.int64, device="cuda")
    st = int(torch.cuda.current_stream().cuda_stream)
    assert fg.polymul(a.data_ptr(), na, b.data_ptr(), nb, c_ref.data_ptr(), st) == 0
    assert fg.polymul_noalloc(a.data_ptr(), na, b.data_ptr(), nb, c_new.data_ptr(), st) == 0
    torch.cuda.synchronize()
    return c_ref.cpu().numpy(), c_new.cpu().numpy()


def test_noalloc_exact_on_consecutive_calls(fg):
    g = workloads.generator(1)
    cases = [
        # near the size limit, coefficients in [0, 9]
        (g.integers(0, 10, size=30000, dtype=np.int64),
         g.integers(0, 10, size=35000, dtype=np.int64)),
        # smaller, signed coefficients: finds the first call's values in the
        # shared scratch
        (g.integers(-1000, 1001, size=700, dtype=np.int64),
         g.integers(-1000, 1001, size=1300, dtype=np.int64)),
        # exactly at the limit: na + nb - 1 = FFT_POLYMUL_NOALLOC_MAX_LEN
        (g.integers(-9, 10, size=fg.POLYMUL_NOALLOC_MAX_LEN // 2, dtype=np.int64),
         g.integers(-9, 10, size=fg.POLYMUL_NOALLOC_MAX_LEN // 2 + 1, dtype=np.int64)),
        # the shortest product
        (np.array([7], np.int64), np.array([-3], np.int64)),
    ]
    for a, b in cases:
        ref, new = _both(fg, a, b)
        exact = oracle.polymul_schoolbook(a, b)
        assert np.array_equal(new, exact), (a.size, b.size)
        assert np.array_equal(new, ref), (a.size, b.size)


def test_noalloc_rejects_products_beyond_its_scratch(fg):
    n = fg.POLYMUL_NOALLOC_MAX_LEN // 2 + 1
    a = torch.zeros(n, dtype=torch.int64, device="cuda")
    c = torch.zeros(2 * n - 1, dtype=torch.int64, device="cuda")
    st = int(torch.cuda.current_stream().cuda_stream)
    assert fg.polymul_noalloc(a.data_ptr(), n, a.data_ptr(), n, c.data_ptr(), st) == \
        fg.FFT_ERR_UNSUPPORTED
