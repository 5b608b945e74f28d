"""polymul_noalloc: the polynomial product for callers that cannot allocate
device memory where they need it (a plug-in inside a host application that
owns the memory budget, a latency-critical loop).  Its scratch is a fixed
array inside the library, so its result must equal the allocating entry
point's bit for bit, also on a second call that finds the first call's data
still in that array.  Kept in its own file, collected last."""
import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg(fg_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fg_lib


def _both(fg, na, nb, seed):
    g = workloads.generator(seed)
    a = torch.from_numpy(g.integers(0, 10, size=na, dtype=np.int64)).cuda()
    b = torch.from_numpy(g.integers(0, 10, size=nb, dtype=np.int64)).cuda()
    c_ref = torch.empty(na + nb - 1, dtype=torch.int64, device="cuda")
    c_new = torch.full((na + nb - 1,), -1, dtype=torch.int64, device="cuda")
    st = int(torch.cuda.current_stream().cuda_stream)
    assert fg.polymul(a.data_ptr(), na, b.data_ptr(), nb, c_ref.data_ptr(), st) == 0
    assert fg.polymul_noalloc(a.data_ptr(), na, b.data_ptr(), nb, c_new.data_ptr(), st) == 0
    torch.cuda.synchronize()
    return c_ref.cpu().numpy(), c_new.cpu().numpy()


def test_noalloc_matches_polymul_on_two_calls(fg):
    # First call near the size limit, second smaller: the second finds the
    # first call's values in the shared scratch.
    ref1, new1 = _both(fg, 30000, 35000, 1)
    assert np.array_equal(new1, ref1)
    ref2, new2 = _both(fg, 700, 1300, 2)
    assert np.array_equal(new2, ref2)


def test_noalloc_rejects_products_beyond_its_scratch(fg):
    n = fg.POLYMUL_NOALLOC_MAX_LEN // 2 + 1
    a = torch.zeros(n, dtype=torch.int64, device="cuda")
    c = torch.zeros(2 * n - 1, dtype=torch.int64, device="cuda")
    st = int(torch.cuda.current_stream().cuda_stream)
    assert fg.polymul_noalloc(a.data_ptr(), n, a.data_ptr(), n, c.data_ptr(), st) == \
        fg.FFT_ERR_UNSUPPORTED
