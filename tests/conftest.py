import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large sizes (still bounded)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def build_library():
    """Build libfftgb300.so in-tree if stale (loaded by path: importing the
    package needs the built library)."""
    import importlib.util
    path = os.path.join(ROOT, "fft_convolution_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("fft_convolution_gb300_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


@pytest.fixture(scope="session")
def fg_lib():
    build_library()
    import fft_convolution_gb300
    return fft_convolution_gb300


@pytest.fixture
def opt(fg_lib):
    """Forces library choices through the test hook fft_debug_set_option for
    one test: opt("PASS_SPLIT", "12,10"), opt("NO_CLUSTER", 1), ...; the
    library's own choices are restored afterwards."""
    used = []

    def set_option(name, value):
        code = getattr(fg_lib, "FFT_OPT_" + name)
        if name == "PASS_SPLIT" and isinstance(value, str):
            value = fg_lib.pass_split_value(int(v) for v in value.split(","))
        assert fg_lib.fft_debug_set_option(code, int(value)) == fg_lib.FFT_OK, (name, value)
        used.append(code)
    yield set_option
    for code in used:
        fg_lib.fft_debug_set_option(code, -1)
