"""Python binding of the GB300 power-of-two FFT library (``libfftgb300.so``).

A thin ctypes layer over the C ABI of ``include/fft_gb300.h``: the functions
below carry the same names and arguments and only marshal them; every step
of every transform runs in the library's CUDA kernels.  PyTorch is used only
for device memory and streams (the tensor helpers at the end).

Importing this package loads the in-tree shared library and raises
``ImportError`` if it has not been built (``python
fft_convolution_gb300/build.py``); there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfftgb300.so")

FFT_OK = 0
FFT_ERR_INVALID_ARG = 1
FFT_ERR_NOT_POW2 = 2
FFT_ERR_UNSUPPORTED = 3
FFT_ERR_CUDA = 4
FFT_ERR_ALLOC = 5
FFT_ERR_MISALIGNED = 6
FFT_ERR_DEVICE_TIMEOUT = 7

FFT_FORWARD = -1
FFT_INVERSE = +1

FFT_C2C_F32 = 0
FFT_C2C_F64 = 1
FFT_REAL_F32 = 2
FFT_REAL_F64 = 3

FFT_CONV_COMPLEX = 0
FFT_CONV_REAL = 1

FFT_OPT_PASS_LOG = 1
FFT_OPT_PASS_SPLIT = 2
FFT_OPT_NO_TMA = 3
FFT_OPT_NO_CLUSTER = 4
FFT_OPT_CLUSTER_LOG_MIN = 5
FFT_OPT_ND_ROWS_T = 6
FFT_OPT_COL_RADIX_LOG = 7
FFT_OPT_ROWS_SHFL = 8
FFT_OPT_PASS_SHFL = 9

# Every symbol the header declares, with its ctypes signature.
_VP, _I64, _INT, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "fft_plan_create": (_VP, [_I64, _I64, _INT, _INT, _INT]),
    "fft_plan_create_nd": (_VP, [_INT, _VP, _I64, _INT, _INT]),
    "fft_plan_destroy": (None, [_VP]),
    "fft_plan_workspace_bytes": (_SZ, [_VP]),
    "fft_plan_num_kernels": (_INT, [_VP]),
    "fft_exec": (_INT, [_VP, _VP, _VP, _VP]),
    "fft_exec_host": (_INT, [_VP, _VP, _VP, _VP, _VP, _VP]),
    "fft_exec_host_chain": (_INT, [_VP, _INT, _VP, _VP, _VP, _VP, _I64, _VP]),
    "polymul": (_INT, [_VP, _I64, _VP, _I64, _VP, _VP]),
    "polymul_batched": (_INT, [_VP, _I64, _VP, _I64, _VP, _I64, _VP]),
    "polymul_batched_host": (_INT, [_VP, _I64, _VP, _I64, _VP, _I64, _VP, _VP, _VP, _I64, _VP]),
    "polymul_noalloc": (_INT, [_VP, _I64, _VP, _I64, _VP, _VP]),
    "polymul_num_kernels": (_INT, [_I64, _I64]),
    "fft_convolve": (_INT, [_VP, _I64, _VP, _I64, _VP, _I64, _INT, _INT, _INT, _VP]),
    "fft_convolve_num_kernels": (_INT, [_I64, _I64, _I64, _INT, _INT, _INT]),
    "fft_convolve_host": (_INT, [_VP, _I64, _VP, _I64, _VP, _I64, _INT, _INT, _INT, _VP, _VP,
                                 _I64, _VP]),
    "fft_debug_radix2_pass": (_INT, [_VP, _VP, _I64, _I64, _INT, _VP]),
    "fft_device_status": (_INT, [_VP]),
    "fft_debug_wait_timeout": (_INT, [_I64, _VP]),
    "fft_debug_cluster_timeout": (_INT, [_VP, _I64, _VP]),
    "fft_debug_set_option": (_INT, [_INT, _I64]),
    "fft_last_status": (_INT, []),
    "fft_status_string": (ctypes.c_char_p, [_INT]),
    "fft_last_cuda_error": (ctypes.c_char_p, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python fft_convolution_gb300/build.py); there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


class FFTError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = fft_status_string(status)
        if status == FFT_ERR_CUDA or status == FFT_ERR_ALLOC:
            msg += f" ({fft_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [status {status}]")
        self.status = status


def _check(rc: int, what: str) -> None:
    if rc != FFT_OK:
        raise FFTError(rc, what)


# ---- the C ABI, name for name -------------------------------------------------

def fft_plan_create(n: int, batch: int, dims: int, direction: int, dtype: int) -> int:
    """Returns the plan handle; raises FFTError with fft_last_status()."""
    h = _lib.fft_plan_create(n, batch, dims, direction, dtype)
    if not h:
        raise FFTError(_lib.fft_last_status(), "fft_plan_create")
    return h


def fft_plan_create_nd(rank: int, shape, batch: int, direction: int, dtype: int) -> int:
    """shape: a sequence of `rank` sides (marshalled to an int64 array)."""
    arr = (ctypes.c_int64 * rank)(*shape)
    h = _lib.fft_plan_create_nd(rank, arr, batch, direction, dtype)
    if not h:
        raise FFTError(_lib.fft_last_status(), "fft_plan_create_nd")
    return h


def fft_plan_destroy(plan: int) -> None:
    _lib.fft_plan_destroy(plan)


def fft_plan_workspace_bytes(plan: int) -> int:
    return int(_lib.fft_plan_workspace_bytes(plan))


def fft_plan_num_kernels(plan: int) -> int:
    return int(_lib.fft_plan_num_kernels(plan))


def fft_exec(plan: int, in_ptr: int, out_ptr: int, stream: int) -> int:
    return _lib.fft_exec(plan, in_ptr, out_ptr, stream)


def fft_exec_host(plan: int, host_in: int, host_out: int, dev_in: int, dev_out: int,
                  stream: int) -> int:
    return _lib.fft_exec_host(plan, host_in, host_out, dev_in, dev_out, stream)


def fft_exec_host_chain(plans, nplans: int, host_in: int, host_out: int, dev_a: int, dev_b: int,
                        chunk: int, stream: int) -> int:
    """plans: a sequence of plan handles (marshalled to a C array)."""
    arr = (ctypes.c_void_p * len(plans))(*plans)
    return _lib.fft_exec_host_chain(arr, nplans, host_in, host_out, dev_a, dev_b, chunk, stream)


def polymul(a_ptr: int, na: int, b_ptr: int, nb: int, c_ptr: int, stream: int) -> int:
    return _lib.polymul(a_ptr, na, b_ptr, nb, c_ptr, stream)


def polymul_batched(a_ptr: int, na: int, b_ptr: int, nb: int, c_ptr: int, batch: int,
                    stream: int) -> int:
    return _lib.polymul_batched(a_ptr, na, b_ptr, nb, c_ptr, batch, stream)


def polymul_batched_host(a_host: int, na: int, b_host: int, nb: int, c_host: int, batch: int,
                         dev_a: int, dev_b: int, dev_c: int, chunk: int, stream: int) -> int:
    return _lib.polymul_batched_host(a_host, na, b_host, nb, c_host, batch, dev_a, dev_b, dev_c,
                                     chunk, stream)


def polymul_noalloc(a_ptr: int, na: int, b_ptr: int, nb: int, c_ptr: int, stream: int) -> int:
    """polymul without device allocation (fixed scratch; na+nb-1 <=
    POLYMUL_NOALLOC_MAX_LEN).  For callers that may not allocate."""
    return _lib.polymul_noalloc(a_ptr, na, b_ptr, nb, c_ptr, stream)


POLYMUL_NOALLOC_MAX_LEN = 65536


def polymul_num_kernels(na: int, nb: int) -> int:
    return int(_lib.polymul_num_kernels(na, nb))


def fft_convolve(x_ptr: int, nx: int, h_ptr: int, nh: int, y_ptr: int, batch: int,
                 h_per_row: int, kind: int, dtype: int, stream: int) -> int:
    return _lib.fft_convolve(x_ptr, nx, h_ptr, nh, y_ptr, batch, h_per_row, kind, dtype, stream)


def fft_convolve_host(x_host: int, nx: int, h_ptr: int, nh: int, y_host: int, batch: int,
                      h_per_row: int, kind: int, dtype: int, dev_x: int, dev_y: int, chunk: int,
                      stream: int) -> int:
    return _lib.fft_convolve_host(x_host, nx, h_ptr, nh, y_host, batch, h_per_row, kind, dtype,
                                  dev_x, dev_y, chunk, stream)


def fft_convolve_num_kernels(nx: int, nh: int, batch: int, h_per_row: int, kind: int,
                             dtype: int) -> int:
    return int(_lib.fft_convolve_num_kernels(nx, nh, batch, h_per_row, kind, dtype))


def fft_debug_radix2_pass(in_ptr: int, out_ptr: int, n: int, half: int, dtype: int,
                          stream: int) -> int:
    return _lib.fft_debug_radix2_pass(in_ptr, out_ptr, n, half, dtype, stream)


def fft_debug_wait_timeout(polls: int, stream: int) -> int:
    return int(_lib.fft_debug_wait_timeout(polls, stream))


def fft_debug_cluster_timeout(data_ptr: int, polls: int, stream: int) -> int:
    return int(_lib.fft_debug_cluster_timeout(data_ptr, polls, stream))


def fft_debug_set_option(option: int, value: int) -> int:
    """Test / tuning hook: force one planning or launch choice (FFT_OPT_*);
    value < 0 restores the library's own choice."""
    return int(_lib.fft_debug_set_option(option, value))


def pass_split_value(factors) -> int:
    """FFT_OPT_PASS_SPLIT value of a list of per-pass factors (log2), first
    pass first."""
    v = 0
    for k, f in enumerate(factors):
        v |= int(f) << (4 * k)
    return v


def fft_device_status(stream: int) -> int:
    return int(_lib.fft_device_status(stream))


def fft_last_status() -> int:
    return int(_lib.fft_last_status())


def fft_status_string(status: int) -> str:
    return _lib.fft_status_string(status).decode()


def fft_last_cuda_error() -> str:
    return _lib.fft_last_cuda_error().decode()


# ---- torch tensor helpers (allocation and streams only) ------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.complex64:
        return FFT_C2C_F32
    if t.dtype == torch.complex128:
        return FFT_C2C_F64
    raise TypeError(f"expected complex64 or complex128, got {t.dtype}")


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class Plan:
    """Owns one fft_plan handle: `batch` transforms of length n (dims=1)
    or of n x n images (dims=2)."""

    def __init__(self, n: int, batch: int = 1, dims: int = 1, direction: int = FFT_FORWARD,
                 dtype: int = FFT_C2C_F32, shape=None):
        """n / dims as fft_plan_create; or shape=(H, W) / (D, H, W) for
        fft_plan_create_nd."""
        self.batch, self.direction, self.dtype = batch, direction, dtype
        if shape is not None:
            self.shape = tuple(int(v) for v in shape)
            self.handle = fft_plan_create_nd(len(self.shape), self.shape, batch, direction, dtype)
        else:
            self.shape = (n,) if dims == 1 else (n, n)
            self.handle = fft_plan_create(n, batch, dims, direction, dtype)
        self.n, self.dims = self.shape[-1], len(self.shape)

    @property
    def workspace_bytes(self) -> int:
        return fft_plan_workspace_bytes(self.handle)

    @property
    def num_kernels(self) -> int:
        return fft_plan_num_kernels(self.handle)

    def numel(self) -> int:
        total = self.batch
        for v in self.shape:
            total *= v
        return total

    @property
    def real(self) -> bool:
        return self.dtype in (FFT_REAL_F32, FFT_REAL_F64)

    def io_spec(self):
        """((input torch dtype, elements), (output torch dtype, elements))."""
        torch = _torch()
        if not self.real:
            t = torch.complex64 if self.dtype == FFT_C2C_F32 else torch.complex128
            return (t, self.numel()), (t, self.numel())
        rt, ct = ((torch.float32, torch.complex64) if self.dtype == FFT_REAL_F32
                  else (torch.float64, torch.complex128))
        samples = (rt, self.batch * self.n)
        bins = (ct, self.batch * (self.n // 2 + 1))
        return (samples, bins) if self.direction == FFT_FORWARD else (bins, samples)

    def exec(self, inp, out=None, stream=None):
        """Run on contiguous device tensors: complex64 / complex128 for
        complex plans; float samples and complex half spectra (n // 2 + 1
        bins per row) for real plans."""
        torch = _torch()
        (it, ni), (ot, no) = self.io_spec()
        if out is None:
            if self.real:
                shape = (self.batch, no // self.batch)
                out = torch.empty(shape, dtype=ot, device=inp.device)
            else:
                out = torch.empty_like(inp)
        if not (inp.is_cuda and out.is_cuda and inp.is_contiguous() and out.is_contiguous()):
            raise ValueError("exec needs contiguous CUDA tensors")
        if inp.numel() != ni or out.numel() != no:
            raise ValueError(f"tensors must hold {ni} and {no} elements")
        if inp.dtype != it or out.dtype != ot:
            raise TypeError("tensor dtype does not match the plan")
        _check(fft_exec(self.handle, inp.data_ptr(), out.data_ptr(), _stream_handle(stream)),
               "fft_exec")
        return out

    def exec_host(self, host_in, host_out, dev_in, dev_out, stream=None):
        """Host-staged run (see fft_exec_host); host tensors should be pinned."""
        hin = host_in.data_ptr() if host_in is not None else None
        hout = host_out.data_ptr() if host_out is not None else None
        _check(fft_exec_host(self.handle, hin, hout, dev_in.data_ptr(), dev_out.data_ptr(),
                             _stream_handle(stream)), "fft_exec_host")

    def chain_host(self, others, host_in, host_out, dev_a, dev_b, chunk: int, stream=None):
        """fft_exec_host_chain over [self] + others on host tensors."""
        plans = [self.handle] + [o.handle for o in others]
        _check(fft_exec_host_chain(plans, len(plans), host_in.data_ptr(), host_out.data_ptr(),
                                   dev_a.data_ptr(), dev_b.data_ptr(), chunk,
                                   _stream_handle(stream)), "fft_exec_host_chain")

    def close(self):
        if getattr(self, "handle", None):
            fft_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fft(x, direction: int = FFT_FORWARD, out=None, stream=None):
    """Transforms along the last axis of a contiguous CUDA tensor."""
    n = x.shape[-1]
    p = Plan(n, x.numel() // n, 1, direction, _dtype_code(x))
    try:
        return p.exec(x, out, stream)
    finally:
        if stream is None:
            _torch().cuda.current_stream().synchronize()
        p.close()


def fft2(x, direction: int = FFT_FORWARD, out=None, stream=None):
    """2D transform of the last two (equal, power-of-two) axes."""
    n = x.shape[-1]
    if x.shape[-2] != n:
        raise ValueError("2D transforms are N x N")
    p = Plan(n, x.numel() // (n * n), 2, direction, _dtype_code(x))
    try:
        return p.exec(x, out, stream)
    finally:
        if stream is None:
            _torch().cuda.current_stream().synchronize()
        p.close()


def polymul_tensors(a, b, out=None, stream=None):
    """c = a * b for int64 CUDA tensors [batch, na] and [batch, nb]
    (or 1D); returns [batch, na+nb-1]."""
    torch = _torch()
    squeeze = a.dim() == 1
    a2 = a.reshape(1, -1) if squeeze else a
    b2 = b.reshape(1, -1) if squeeze else b
    if a2.dtype != torch.int64 or b2.dtype != torch.int64:
        raise TypeError("polymul takes int64 coefficients")
    batch, na = a2.shape
    nb = b2.shape[1]
    if b2.shape[0] != batch:
        raise ValueError("a and b need the same batch")
    if out is None:
        out = torch.empty(batch, na + nb - 1, dtype=torch.int64, device=a.device)
    a2, b2 = a2.contiguous(), b2.contiguous()
    _check(polymul_batched(a2.data_ptr(), na, b2.data_ptr(), nb, out.data_ptr(), batch,
                           _stream_handle(stream)), "polymul_batched")
    return out.reshape(-1) if squeeze else out


def convolve(x, h, out=None, stream=None):
    """Linear convolution of every row of x (CUDA tensor [batch, nx] or
    [nx]; float32 / float64 / complex64 / complex128) with h ([nh] shared,
    or [batch, nh] per row, same dtype); returns [batch, nx + nh - 1]."""
    torch = _torch()
    kinds = {torch.float32: (FFT_CONV_REAL, FFT_C2C_F32), torch.float64: (FFT_CONV_REAL, FFT_C2C_F64),
             torch.complex64: (FFT_CONV_COMPLEX, FFT_C2C_F32),
             torch.complex128: (FFT_CONV_COMPLEX, FFT_C2C_F64)}
    if x.dtype not in kinds or h.dtype != x.dtype:
        raise TypeError("x and h must share one of float32/64, complex64/128")
    kind, dtype = kinds[x.dtype]
    squeeze = x.dim() == 1
    x2 = (x.reshape(1, -1) if squeeze else x).contiguous()
    batch, nx = x2.shape
    h_per_row = 1 if h.dim() == 2 else 0
    h2 = h.contiguous()
    nh = h2.shape[-1]
    if h_per_row and h2.shape[0] != batch:
        raise ValueError("a per-row filter needs one row per signal")
    if out is None:
        out = torch.empty(batch, nx + nh - 1, dtype=x.dtype, device=x.device)
    _check(fft_convolve(x2.data_ptr(), nx, h2.data_ptr(), nh, out.data_ptr(), batch, h_per_row,
                        kind, dtype, _stream_handle(stream)), "fft_convolve")
    return out.reshape(-1) if squeeze else out


def rfft(x, out=None, stream=None):
    """Half spectra (n // 2 + 1 bins) of the real rows along the last axis of
    a contiguous float32 / float64 CUDA tensor."""
    torch = _torch()
    if x.dtype not in (torch.float32, torch.float64):
        raise TypeError("rfft takes float32 or float64 samples")
    n = x.shape[-1]
    p = Plan(n, x.numel() // n, 1, FFT_FORWARD,
             FFT_REAL_F32 if x.dtype == torch.float32 else FFT_REAL_F64)
    try:
        y = p.exec(x, out, stream)
        return y.reshape(tuple(x.shape[:-1]) + (n // 2 + 1,))
    finally:
        if stream is None:
            torch.cuda.current_stream().synchronize()
        p.close()


def irfft(X, n: int, out=None, stream=None):
    """Real rows of length n from half spectra (n // 2 + 1 bins, complex64 /
    complex128 CUDA tensor, last axis), scaled by 1/n."""
    torch = _torch()
    if X.shape[-1] != n // 2 + 1:
        raise ValueError("the last axis must hold n // 2 + 1 bins")
    dt = _dtype_code(X)
    p = Plan(n, X.numel() // X.shape[-1], 1, FFT_INVERSE,
             FFT_REAL_F32 if dt == FFT_C2C_F32 else FFT_REAL_F64)
    try:
        y = p.exec(X, out, stream)
        return y.reshape(tuple(X.shape[:-1]) + (n,))
    finally:
        if stream is None:
            torch.cuda.current_stream().synchronize()
        p.close()


def fftn(x, ndim: int, direction: int = FFT_FORWARD, out=None, stream=None):
    """Transforms over the last `ndim` (1-3) axes of a contiguous CUDA
    tensor, sides of any length."""
    shape = tuple(x.shape[-ndim:])
    batch = x.numel()
    for v in shape:
        batch //= v
    p = Plan(0, batch, direction=direction, dtype=_dtype_code(x), shape=shape)
    try:
        return p.exec(x, out, stream)
    finally:
        if stream is None:
            _torch().cuda.current_stream().synchronize()
        p.close()
