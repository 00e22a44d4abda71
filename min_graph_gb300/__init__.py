"""min_graph_gb300 -- Python binding of libapsp, all-pairs shortest paths by
blocked Floyd-Warshall on one GB300 GPU (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libapsp.so (built by min_graph_gb300.build).  PyTorch supplies
device memory and streams.  There is no CPU fallback: if the library is
missing, every call raises.

    import torch, min_graph_gb300 as apsp
    d = torch.full((n, n), apsp.INF_I32, dtype=torch.int32, device="cuda")
    ...fill arcs, zero diagonal...
    apsp.solve(d)                 # in place, asynchronous on the current stream

The functions mirror the C-ABI in include/apsp.h (same names without the
apsp_ prefix).
"""
from __future__ import annotations

import ctypes
import os
import threading

INF_I32 = 0x3FFFFFFF
TILE = 128
MAX_N = 262144

OK, EINVAL, ECUDA, ETIMEOUT, EUNSUPPORTED, ENOMEM = range(6)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libapsp.so")
_lock = threading.Lock()
_lib = None


class ApspError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {status_string(status)}"
        if status == ECUDA and _lib is not None:
            msg += f" (cudaError {_lib.apsp_last_cuda_error()})"
        super().__init__(msg)


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libapsp.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libapsp.so not found at {_LIB_PATH}; build it with "
                "`python -m min_graph_gb300.build` (the library has no CPU fallback)")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        for name in ("apsp_solve", "apsp_solve_i32", "apsp_solve_f32",
                     "apsp_solve_host_i32", "apsp_solve_host_f32"):
            f = getattr(lib, name)
            f.argtypes = [vp, i32, i32, vp]
            f.restype = i32
        for name in ("apsp_validate_i32", "apsp_validate_f32"):
            f = getattr(lib, name)
            f.argtypes = [vp, i32, i32, vp, vp]
            f.restype = i32
        lib.apsp_stream_check.argtypes = [vp]
        lib.apsp_stream_check.restype = i32
        lib.apsp_last_cuda_error.argtypes = []
        lib.apsp_last_cuda_error.restype = i32
        lib.apsp_status_string.argtypes = [i32]
        lib.apsp_status_string.restype = ctypes.c_char_p
        lib.apsp_version.argtypes = []
        lib.apsp_version.restype = i32
        lib.apsp_release.argtypes = []
        lib.apsp_release.restype = i32
        lib.apsp_phase_timing_enable.argtypes = [i32]
        lib.apsp_phase_timing_enable.restype = i32
        lib.apsp_phase_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]
        lib.apsp_phase_timing_read.restype = i32
        lib.apsp_debug_inject_phase3_timeout.argtypes = [ctypes.c_ulonglong]
        lib.apsp_debug_inject_phase3_timeout.restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    lib = _lib if _lib is not None else load()
    return lib.apsp_status_string(int(status)).decode()


def version() -> int:
    return load().apsp_version()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise ApspError(status, what)


def _stream_handle(t, stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _matrix_args(t):
    """(pointer, n, ld) of a square 2-D CUDA tensor with unit column stride."""
    import torch

    if not isinstance(t, torch.Tensor) or t.dim() != 2 or t.shape[0] != t.shape[1]:
        raise ValueError("expected a square 2-D tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor (use solve_host for host memory)")
    n = int(t.shape[0])
    if n > 1 and t.stride(1) != 1:
        raise ValueError("the column stride must be 1 (row-major matrix)")
    ld = int(t.stride(0)) if n > 1 else max(1, n)
    return t.data_ptr(), n, ld


def solve(t, stream=None):
    """In-place APSP on a square int32 or float32 CUDA tensor (row-major,
    leading dimension = t.stride(0)).  Asynchronous on `stream` (default:
    the current stream).  Returns t."""
    import torch

    lib = load()
    ptr, n, ld = _matrix_args(t)
    s = _stream_handle(t, stream)
    with torch.cuda.device(t.device):
        if t.dtype == torch.int32:
            _check(lib.apsp_solve(ptr, n, ld, s), "apsp_solve")
        elif t.dtype == torch.float32:
            _check(lib.apsp_solve_f32(ptr, n, ld, s), "apsp_solve_f32")
        else:
            raise TypeError("dtype must be int32 or float32")
    return t


def solve_host(a, n: int | None = None, ld: int | None = None, stream=None):
    """End-to-end APSP on a HOST matrix (numpy array or CPU tensor, ideally
    pinned): the library copies it to the device, solves, copies the result
    back in place and waits.  Uses the current CUDA device."""
    import numpy as np
    import torch

    lib = load()
    if isinstance(a, torch.Tensor):
        if a.is_cuda or a.dim() != 2 or (a.shape[0] > 1 and a.stride(1) != 1):
            raise ValueError("expected a row-major 2-D CPU tensor")
        ptr, rows, ld0, dt = a.data_ptr(), a.shape[0], a.stride(0), a.dtype
        is_i32, is_f32 = dt == torch.int32, dt == torch.float32
    else:
        if not isinstance(a, np.ndarray) or a.ndim != 2 or not a.flags.c_contiguous:
            raise ValueError("expected a C-contiguous 2-D numpy array")
        ptr, rows, ld0 = a.ctypes.data, a.shape[0], a.shape[1]
        is_i32, is_f32 = a.dtype == np.int32, a.dtype == np.float32
    n = rows if n is None else n
    ld = ld0 if ld is None else ld
    if n > rows or ld != ld0:
        raise ValueError("n / ld do not match the array")
    s = 0 if stream is None else (int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))
    if is_i32:
        _check(lib.apsp_solve_host_i32(ptr, n, ld, s), "apsp_solve_host_i32")
    elif is_f32:
        _check(lib.apsp_solve_host_f32(ptr, n, ld, s), "apsp_solve_host_f32")
    else:
        raise TypeError("dtype must be int32 or float32")
    return a


def validate(t, stream=None) -> int:
    """Check the preconditions on the device; returns the flag bits
    (1 non-zero diagonal, 2 negative entry, 4 NaN).  Synchronises."""
    import torch

    lib = load()
    ptr, n, ld = _matrix_args(t)
    s = _stream_handle(t, stream)
    flags = torch.zeros(1, dtype=torch.int32, device=t.device)
    with torch.cuda.device(t.device):
        if t.dtype == torch.int32:
            _check(lib.apsp_validate_i32(ptr, n, ld, s, flags.data_ptr()), "apsp_validate_i32")
        elif t.dtype == torch.float32:
            _check(lib.apsp_validate_f32(ptr, n, ld, s, flags.data_ptr()), "apsp_validate_f32")
        else:
            raise TypeError("dtype must be int32 or float32")
        stream_check(s)
    return int(flags.item())


def stream_check(stream=None) -> None:
    """Wait for the stream and raise on any error from its work."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    s = int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)
    _check(load().apsp_stream_check(s), "apsp_stream_check")


def release() -> None:
    _check(load().apsp_release(), "apsp_release")


def phase_timing_enable(enable: bool = True) -> None:
    _check(load().apsp_phase_timing_enable(int(bool(enable))), "apsp_phase_timing_enable")


def phase_timing_read():
    """Returns ([ms phase1, ms phase2, ms phase3], [launches...]) since the
    last read.  Waits for the recorded events."""
    ms = (ctypes.c_double * 3)()
    cnt = (ctypes.c_longlong * 3)()
    _check(load().apsp_phase_timing_read(ms, cnt), "apsp_phase_timing_read")
    return list(ms), list(cnt)


def debug_inject_phase3_timeout(timeout_ns: int) -> None:
    """Test hook (include/apsp_debug.h): the next solve that runs the
    persistent phase 3 skips one k-slab, so a bounded device wait runs out
    after `timeout_ns` and the next stream_check raises ApspError(ETIMEOUT)."""
    _check(load().apsp_debug_inject_phase3_timeout(int(timeout_ns)), "apsp_debug_inject_phase3_timeout")
