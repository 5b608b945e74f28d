"""CPU checks of the C ABI: the library loads, exports every symbol the
header declares, and its host-side argument checks answer without a GPU
(no kernel is launched by any call here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fft_gb300.h")


@pytest.fixture(scope="module")
def fg(fg_lib):
    return fg_lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_abi():
    names = declared_functions()
    for want in ("fft_plan_create", "fft_exec", "polymul", "polymul_batched",
                 "fft_plan_destroy", "fft_debug_radix2_pass", "fft_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(fg):
    lib = ctypes.CDLL(fg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fg.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if " T " in line)
    assert exported == set(declared_functions())


def test_binding_covers_the_header(fg):
    assert set(fg.SIGNATURES) == set(declared_functions())
    for name in declared_functions():
        assert callable(getattr(fg, name))


def test_binding_constants_match_the_header(fg):
    # Every numeric #define of the header has the same value in the binding
    # (FFT_POLYMUL_NOALLOC_MAX_LEN is POLYMUL_NOALLOC_MAX_LEN there), so a
    # test that uses the binding's constant checks the library's limit.
    text = open(HEADER).read()
    defines = re.findall(r"^#define\s+(FFT_\w+)\s+\(?([+-]?\d+)\)?", text, flags=re.M)
    assert len(defines) >= 15
    for name, value in defines:
        py_name = "POLYMUL_NOALLOC_MAX_LEN" if name == "FFT_POLYMUL_NOALLOC_MAX_LEN" else name
        assert getattr(fg, py_name) == int(value), name


def test_status_strings(fg):
    assert fg.fft_status_string(0) == "ok"
    for code in range(1, 7):
        assert fg.fft_status_string(code) not in ("ok", "unknown status")
    assert fg.fft_status_string(99) == "unknown status"


@pytest.mark.parametrize("args,status", [
    ((0, 1, 1, -1, 0), 1),        # n <= 0
    ((8, 0, 1, -1, 0), 1),        # batch <= 0
    ((8, 1, 3, -1, 0), 1),        # dims
    ((8, 1, 1, 0, 0), 1),         # direction
    ((8, 1, 1, -1, 7), 1),        # dtype
    ((1 << 31, 1, 2, 1, 1), 3),   # 2D side beyond 2^30
    ((1 << 21, 1 << 20, 2, -1, 0), 3),  # more than 2^40 elements
    ((1 << 31, 1, 1, -1, 0), 3),  # 1D beyond the supported length
])
def test_plan_create_rejects(fg, args, status):
    h = fg._lib.fft_plan_create(*args)
    assert not h
    assert fg.fft_last_status() == status


@pytest.mark.parametrize("n,dims,dtype,kernels", [
    (1, 1, 0, 1), (1024, 1, 0, 1), (1 << 14, 1, 0, 1), (1 << 13, 1, 1, 1),
    (12, 1, 0, 1), (63, 1, 1, 1),  # short non-power-of-two lengths: the direct DFT
    (1, 2, 0, 1)])
def test_on_chip_plans_need_no_device(fg, n, dims, dtype, kernels):
    # Single-kernel plans own no workspace, so they are created without
    # touching the device.  (2D plans of power-of-two sides own one for their
    # transposed-store passes.)
    h = fg._lib.fft_plan_create(n, 3, dims, -1, dtype)
    assert h
    assert fg.fft_plan_num_kernels(h) == kernels
    assert fg.fft_plan_workspace_bytes(h) == 0
    fg.fft_plan_destroy(h)


def test_debug_set_option_checks(fg):
    # The test / tuning hook validates its arguments and restores defaults
    # with a negative value.
    assert fg.fft_debug_set_option(99, 1) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_set_option(0, 1) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_set_option(fg.FFT_OPT_PASS_LOG, 3) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_set_option(fg.FFT_OPT_CLUSTER_LOG_MIN, 10) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_set_option(fg.FFT_OPT_COL_RADIX_LOG, 4) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_set_option(fg.FFT_OPT_NO_TMA, 2) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_set_option(fg.FFT_OPT_ROWS_SHFL, 2) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_set_option(fg.FFT_OPT_PASS_SHFL, 2) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_set_option(fg.FFT_OPT_PASS_SHFL + 1, 0) == fg.FFT_ERR_INVALID_ARG
    for code in range(1, fg.FFT_OPT_PASS_SHFL + 1):
        assert fg.fft_debug_set_option(code, -1) == fg.FFT_OK
    assert fg.pass_split_value([9, 9, 8]) == 9 | 9 << 4 | 8 << 8


def test_2d_folded_column_radix_keeps_two_kernels(fg, opt):
    # 2048 x 2048: rows (with the column transform's first radix-4 stage)
    # and one column pass, with or without the fold; no workspace either way.
    for logr in (-1, 0, 1, 2, 3):
        if logr >= 0:
            opt("COL_RADIX_LOG", logr)
        h = fg._lib.fft_plan_create(2048, 3, 2, -1, 0)
        assert h
        assert fg.fft_plan_num_kernels(h) == 2
        assert fg.fft_plan_workspace_bytes(h) == 0
        fg.fft_plan_destroy(h)


def test_exec_argument_checks(fg):
    h = fg._lib.fft_plan_create(64, 1, 1, -1, 0)
    assert h
    assert fg.fft_exec(h, None, 16, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_exec(None, 16, 16, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_exec(h, 16 + 8, 32, None) == fg.FFT_ERR_MISALIGNED
    assert fg.fft_exec(h, 16, 32 + 4, None) == fg.FFT_ERR_MISALIGNED
    assert fg.fft_exec_host(h, None, None, None, 16, None) == fg.FFT_ERR_INVALID_ARG
    fg.fft_plan_destroy(h)
    fg.fft_plan_destroy(None)


def test_polymul_and_debug_argument_checks(fg):
    assert fg.polymul(16, 0, 16, 4, 16, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.polymul(None, 4, 16, 4, 16, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.polymul(20, 4, 16, 4, 16, None) == fg.FFT_ERR_MISALIGNED
    assert fg.polymul(16, 1 << 27, 16, 1 << 27, 16, None) == fg.FFT_ERR_UNSUPPORTED
    assert fg.polymul_batched(16, 4, 16, 4, 16, 0, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_radix2_pass(16, 32, 8, 3, 0, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_radix2_pass(16, 32, 8, 0, 0, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_radix2_pass(16, 32, 8, 2, 5, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_radix2_pass(24, 32, 8, 2, 0, None) == fg.FFT_ERR_MISALIGNED
    assert fg.fft_debug_cluster_timeout(None, 10, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_cluster_timeout(16, 0, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_cluster_timeout(16, (1 << 22) + 1, None) == fg.FFT_ERR_INVALID_ARG
    assert fg.fft_debug_cluster_timeout(24, 10, None) == fg.FFT_ERR_MISALIGNED


@pytest.mark.parametrize("n,dtype", [(2, 2), (8, 2), (4096, 2), (1 << 15, 2), (1 << 14, 3), (2, 3)])
def test_on_chip_real_plans_need_no_device(fg, n, dtype):
    # n = 2H with H a power of two on chip: one kernel each way, no workspace.
    for direction in (-1, 1):
        h = fg._lib.fft_plan_create(n, 5, 1, direction, dtype)
        assert h, fg.fft_last_status()
        assert fg.fft_plan_num_kernels(h) == 1
        assert fg.fft_plan_workspace_bytes(h) == 0
        fg.fft_plan_destroy(h)


def test_real_plan_argument_checks(fg):
    assert not fg._lib.fft_plan_create(64, 1, 2, -1, fg.FFT_REAL_F32)
    assert fg.fft_last_status() == fg.FFT_ERR_UNSUPPORTED
    h = fg._lib.fft_plan_create(64, 1, 1, -1, fg.FFT_REAL_F32)
    assert h
    assert fg.fft_exec(h, 16, 16, None) == fg.FFT_ERR_INVALID_ARG  # in place
    assert fg.fft_exec(h, 16 + 8, 32, None) == fg.FFT_ERR_MISALIGNED
    fg.fft_plan_destroy(h)
