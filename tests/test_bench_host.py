"""Host logic of bench.py, on the CPU: the inputs it synthesises for reduced
profiling shapes match the batch the plans are created with (a mismatch
would hand the library buffers smaller than the plan reads), and the byte
accounting behind the roofline figures."""
import numpy as np
import pytest

import bench


@pytest.fixture(autouse=True)
def _clear_override():
    bench.SIZE_OVERRIDE.clear()
    yield
    bench.SIZE_OVERRIDE.clear()


@pytest.mark.parametrize("name,override,shape", [
    ("c3", dict(n=1 << 12, batch=4), (4, 1 << 12)),
    ("c2", dict(n=256, batch=3), (3, 256)),
    ("any1", dict(batch=2), (2, 3000)),
    ("c4", dict(n=64, batch=2), (2, 64, 64)),
    ("real1", dict(n=64, batch=5), (5, 64)),
    ("nd1", dict(batch=2), (2, 128, 256, 256)),
    ("rows512", dict(batch=7), (7, 512)),
])
def test_reduced_inputs_match_the_batch(name, override, shape):
    bench.SIZE_OVERRIDE.update(override)
    x = bench.sized_input(name, bench.config_of(name))
    assert x.shape == shape


def test_c3_reduced_rows_are_distinct_tone_signals():
    bench.SIZE_OVERRIDE.update(n=1 << 10, batch=3)
    x = bench.sized_input("c3", bench.config_of("c3"))
    assert not np.allclose(x[0], x[1])


def test_roofline_byte_accounting():
    gib = 1 << 30
    c2 = bench.workload_info("c2")
    assert c2["passes"] == 1 and c2["bytes_per_step"] == 2 * 2 * 512 * (1 << 20)
    c3 = bench.workload_info("c3", passes=3)
    assert c3["bytes_per_step"] == 3 * gib and c3["min_bytes_per_step"] == 2 * gib
    assert c3["min_passes"] == 2 and c3["ideal_bytes_per_step"] == gib
    c4 = bench.workload_info("c4")
    assert c4["passes"] == 2 and c4["bytes_per_step"] == 2 * 2 * 2 * 256 * (1 << 20)
    c5 = bench.workload_info("c5")
    L = 1 << 21
    assert c5["flops_per_step"] == 3 * 5.0 * L * 21 * 64
    assert c5["fp64_flops_per_step"] == (5.0 * L * 21 + 5.0 * (L // 2) * 20) * 64


def test_traffic_only_for_the_captured_workload():
    # The committed DRAM counters describe each workload at its own size
    # with the library's own choices; a resized run or one with forced
    # options reports none.
    ent = bench.committed_traffic("c2")
    assert ent is not None and ent["traffic_bytes_per_launch"] > 0
    bench.SIZE_OVERRIDE.update(n=1024, batch=4)
    assert bench.committed_traffic("c2") is None
    bench.SIZE_OVERRIDE.clear()
    bench.OPTIONS.append("PASS_SHFL=1")
    try:
        assert bench.committed_traffic("c2") is None
    finally:
        bench.OPTIONS.remove("PASS_SHFL=1")
    assert bench.committed_traffic("c2") is not None


def test_reference_step_is_capped_at_one_full_step():
    # The reference arm runs a whole step when it fits the time budget and
    # never more: c1 is one 1024-point transform, so one unit is the step.
    r = bench.cpu_oracle_sample("c1", budget_s=5.0, threads=2, max_fraction=1.0)
    assert r["step_fraction"] == 1.0
    assert r["sample"].startswith("1 ")
    # Without the cap the same budget runs many steps' worth of units.
    r = bench.cpu_oracle_sample("c1", budget_s=0.2, threads=1)
    assert r["step_fraction"] > 1.0
