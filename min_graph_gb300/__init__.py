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

The functions mirror the C-ABI in include/apsp.h and include/apsp_sparse.h
(same names without the apsp_ prefix).  The sparse entry points (Johnson's
APSP with Delta-stepping searches) also take negative arc weights:

    apsp.solve_sparse(d)          # in place, blocking; ApspError(ENEGCYCLE)
                                  # when there is a negative cycle
"""
from __future__ import annotations

import ctypes
import os
import threading

INF_I32 = 0x3FFFFFFF
TILE = 128
MAX_N = 262144

SPARSE_MAX_N = 32768

OK, EINVAL, ECUDA, ETIMEOUT, EUNSUPPORTED, ENOMEM, ENEGCYCLE = range(7)

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
        for name in ("apsp_solve_host_batch_i32", "apsp_solve_host_batch_f32"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, i32, i32, i32, vp]
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
        lib.apsp_debug_inject_grid_timeout.argtypes = [ctypes.c_ulonglong]
        lib.apsp_debug_inject_grid_timeout.restype = i32
        lib.apsp_debug_fail_next_allocations.argtypes = [i32]
        lib.apsp_debug_fail_next_allocations.restype = i32
        lib.apsp_debug_small_cluster_size.argtypes = [i32]
        lib.apsp_debug_small_cluster_size.restype = i32
        lib.apsp_solve_sparse_i32.argtypes = [vp, i32, i32, i32, vp]
        lib.apsp_solve_sparse_i32.restype = i32
        lib.apsp_johnson_csr_i32.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp]
        lib.apsp_johnson_csr_i32.restype = i32
        lib.apsp_sssp_delta_i32.argtypes = [vp, vp, vp, i32, vp, i32, i32, vp, i32, vp]
        lib.apsp_sssp_delta_i32.restype = i32
        lib.apsp_csr_count_i32.argtypes = [vp, i32, i32, vp, ctypes.POINTER(i64), vp]
        lib.apsp_csr_count_i32.restype = i32
        lib.apsp_csr_fill_i32.argtypes = [vp, i32, i32, vp, vp, vp, vp]
        lib.apsp_csr_fill_i32.restype = i32
        lib.apsp_sparse_release.argtypes = []
        lib.apsp_sparse_release.restype = i32
        lib.apsp_sssp_i32.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        lib.apsp_sssp_i32.restype = i32
        lib.apsp_sssp_graph_create.argtypes = [vp, vp, vp, i32, i32, vp, ctypes.POINTER(vp)]
        lib.apsp_sssp_graph_create.restype = i32
        lib.apsp_sssp_graph_search.argtypes = [vp, i32, vp, vp]
        lib.apsp_sssp_graph_search.restype = i32
        lib.apsp_sssp_graph_info.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(i32)]
        lib.apsp_sssp_graph_info.restype = i32
        lib.apsp_sssp_graph_destroy.argtypes = [vp]
        lib.apsp_sssp_graph_destroy.restype = i32
        u64 = ctypes.c_ulonglong
        for name in ("apsp_solve_ooc_i32", "apsp_solve_ooc_f32"):
            f = getattr(lib, name)
            f.argtypes = [vp, i32, i32, u64, i32, vp]
            f.restype = i32
        lib.apsp_ooc_block.argtypes = [i32, u64, i32]
        lib.apsp_ooc_block.restype = i32
        lib.apsp_sparse_timing_enable.argtypes = [i32]
        lib.apsp_sparse_timing_enable.restype = i32
        lib.apsp_sparse_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64),
                                                ctypes.POINTER(i64)]
        lib.apsp_sparse_timing_read.restype = i32
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


def _host_matrix(a):
    """(pointer, rows, cols, ld, dtype name) of a row-major 2-D host matrix
    (numpy array or CPU tensor)."""
    import numpy as np
    import torch

    if isinstance(a, torch.Tensor):
        if a.is_cuda or a.dim() != 2 or (a.shape[0] > 1 and a.stride(1) != 1):
            raise ValueError("expected a row-major 2-D CPU tensor")
        dt = {torch.int32: "i32", torch.float32: "f32"}.get(a.dtype)
        return a.data_ptr(), a.shape[0], a.shape[1], a.stride(0), dt
    if not isinstance(a, np.ndarray) or a.ndim != 2 or not a.flags.c_contiguous:
        raise ValueError("expected a C-contiguous 2-D numpy array")
    dt = {np.dtype(np.int32): "i32", np.dtype(np.float32): "f32"}.get(a.dtype)
    return a.ctypes.data, a.shape[0], a.shape[1], a.shape[1], dt


def solve_host_batch(inputs, outputs=None, stream=None):
    """Solve several square HOST matrices of one size and dtype (numpy arrays
    or CPU tensors, ideally pinned) with their copies overlapped
    (apsp_solve_host_batch_*): while problem b is solved, problem b + 1 is
    uploaded and problem b - 1 downloaded.  Results go to `outputs` (default:
    in place; an input may appear several times only with distinct outputs).
    Blocking; uses the current CUDA device.  Returns the outputs."""
    inputs = list(inputs)
    outputs = inputs if outputs is None else list(outputs)
    if len(outputs) != len(inputs):
        raise ValueError("inputs and outputs differ in length")
    lib = load()
    if not inputs:
        return outputs
    ins = [_host_matrix(a) for a in inputs]
    outs = [_host_matrix(a) for a in outputs]
    _, n, cols, ld, dt = ins[0]
    for (_, r, c, l, d) in ins + outs:
        if r != n or c != n or l != ld or d != dt:
            raise ValueError("every matrix must be square with the same size, leading dimension and dtype")
    if dt is None:
        raise TypeError("dtype must be int32 or float32")
    count = len(ins)
    in_arr = (ctypes.c_void_p * count)(*[x[0] for x in ins])
    out_arr = (ctypes.c_void_p * count)(*[x[0] for x in outs])
    s = 0 if stream is None else (int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))
    name = "apsp_solve_host_batch_" + dt
    _check(getattr(lib, name)(in_arr, out_arr, count, n, ld, s), name)
    return outputs


def solve_ooc(a, device_bytes: int = 0, block: int = 0, stream=None):
    """Out-of-core APSP on a HOST matrix (numpy array or CPU tensor; pin it
    for overlapped copies), streamed through the GPU in K x K super-blocks
    (include/apsp_ooc.h).  device_bytes caps the device memory used (0: 70%
    of what is free); block is K (0: the largest that fits).  In place,
    blocking.  Returns a."""
    import numpy as np
    import torch

    lib = load()
    if isinstance(a, torch.Tensor):
        if a.is_cuda or a.dim() != 2 or a.shape[0] != a.shape[1] or (a.shape[0] > 1 and a.stride(1) != 1):
            raise ValueError("expected a square row-major CPU tensor")
        ptr, n, ld = a.data_ptr(), a.shape[0], a.stride(0)
        is_i32, is_f32 = a.dtype == torch.int32, a.dtype == torch.float32
    else:
        if not isinstance(a, np.ndarray) or a.ndim != 2 or a.shape[0] != a.shape[1] or not a.flags.c_contiguous:
            raise ValueError("expected a square C-contiguous numpy array")
        ptr, n, ld = a.ctypes.data, a.shape[0], a.shape[1]
        is_i32, is_f32 = a.dtype == np.int32, a.dtype == np.float32
    s = 0 if stream is None else (int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))
    if is_i32:
        _check(lib.apsp_solve_ooc_i32(ptr, n, max(ld, 1), int(device_bytes), int(block), s), "apsp_solve_ooc_i32")
    elif is_f32:
        _check(lib.apsp_solve_ooc_f32(ptr, n, max(ld, 1), int(device_bytes), int(block), s), "apsp_solve_ooc_f32")
    else:
        raise TypeError("dtype must be int32 or float32")
    return a


def ooc_block(n: int, device_bytes: int, elem_bytes: int = 4) -> int:
    """The super-block K that solve_ooc would choose (0: nothing fits)."""
    return load().apsp_ooc_block(int(n), int(device_bytes), int(elem_bytes))


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


def debug_small_cluster_size(is_float: bool = False) -> int:
    """CTAs in the cluster that solves n <= 512 on the current device (16, 8,
    or 0 when neither fits); -1 on an unsupported device."""
    return int(load().apsp_debug_small_cluster_size(1 if is_float else 0))


def debug_inject_phase3_timeout(timeout_ns: int) -> None:
    """Test hook (include/apsp_debug.h): the next solve that runs the
    persistent phase 3 skips one k-slab, so a bounded device wait runs out
    after `timeout_ns` and the next stream_check raises ApspError(ETIMEOUT)."""
    _check(load().apsp_debug_inject_phase3_timeout(int(timeout_ns)), "apsp_debug_inject_phase3_timeout")


# ---------------------------------------------------------------- sparse path


def _i32_matrix(t):
    import torch

    ptr, n, ld = _matrix_args(t)
    if t.dtype != torch.int32:
        raise TypeError("dtype must be int32")
    return ptr, n, ld


def _csr_args(row_ptr, col_idx, w):
    import torch

    if row_ptr.dtype != torch.int64 or col_idx.dtype != torch.int32 or w.dtype != torch.int32:
        raise TypeError("CSR arrays must be int64 row_ptr, int32 col_idx, int32 w")
    for a in (row_ptr, col_idx, w):
        if not a.is_cuda or a.dim() != 1 or not a.is_contiguous():
            raise ValueError("CSR arrays must be contiguous 1-D CUDA tensors")
    if col_idx.numel() != w.numel():
        raise ValueError("col_idx and w differ in length")
    return int(row_ptr.numel()) - 1


def solve_sparse(t, delta: int = 0, stream=None):
    """In-place APSP on a square int32 CUDA tensor by Johnson's method with
    Delta-stepping searches (include/apsp_sparse.h).  Negative arc weights
    are allowed; a negative cycle raises ApspError with status ENEGCYCLE and
    leaves t unchanged.  Blocks until done.  Returns t."""
    import torch

    lib = load()
    ptr, n, ld = _i32_matrix(t)
    s = _stream_handle(t, stream)
    with torch.cuda.device(t.device):
        _check(lib.apsp_solve_sparse_i32(ptr, n, ld, int(delta), s), "apsp_solve_sparse_i32")
    return t


def csr_from_dense(t, stream=None):
    """(row_ptr int64[n+1], col_idx int32[m], w int32[m]) of a dense int32
    CUDA matrix: arcs are the off-diagonal entries below INF."""
    import torch

    lib = load()
    ptr, n, ld = _i32_matrix(t)
    s = _stream_handle(t, stream)
    row_ptr = torch.empty(n + 1, dtype=torch.int64, device=t.device)
    m = ctypes.c_longlong(0)
    with torch.cuda.device(t.device):
        _check(lib.apsp_csr_count_i32(ptr, n, ld, row_ptr.data_ptr(), ctypes.byref(m), s),
               "apsp_csr_count_i32")
        # at least one element each, so that the pointers are valid even when m = 0
        col = torch.empty(max(1, m.value), dtype=torch.int32, device=t.device)
        w = torch.empty(max(1, m.value), dtype=torch.int32, device=t.device)
        _check(lib.apsp_csr_fill_i32(ptr, n, ld, row_ptr.data_ptr(), col.data_ptr(), w.data_ptr(), s),
               "apsp_csr_fill_i32")
    return row_ptr, col[:m.value], w[:m.value]


def johnson_csr(row_ptr, col_idx, w, delta: int = 0, out=None, stream=None):
    """All-pairs distances of a CSR graph (Johnson's method) into an n x n
    int32 CUDA tensor (`out`, or a new one).  Blocks until done."""
    import torch

    lib = load()
    n = _csr_args(row_ptr, col_idx, w)
    if out is None:
        out = torch.empty((n, n), dtype=torch.int32, device=row_ptr.device)
    optr, on, old = _i32_matrix(out)
    if on != n:
        raise ValueError("out must be n x n")
    s = _stream_handle(row_ptr, stream)
    with torch.cuda.device(row_ptr.device):
        _check(lib.apsp_johnson_csr_i32(row_ptr.data_ptr(), col_idx.data_ptr(), w.data_ptr(), n,
                                        int(delta), optr, old, s), "apsp_johnson_csr_i32")
    return out


def sssp_delta(row_ptr, col_idx, w, sources, delta: int = 0, out=None, stream=None):
    """Delta-stepping from each source (int32 CUDA tensor) on a CSR graph
    with weights >= 0.  Returns (or fills) an nsrc x n int32 tensor whose
    row q is the distance vector of sources[q].  Blocks until done."""
    import torch

    lib = load()
    n = _csr_args(row_ptr, col_idx, w)
    if sources.dtype != torch.int32 or not sources.is_cuda or sources.dim() != 1 or not sources.is_contiguous():
        raise ValueError("sources must be a contiguous 1-D int32 CUDA tensor")
    nsrc = int(sources.numel())
    if out is None:
        out = torch.empty((nsrc, n), dtype=torch.int32, device=row_ptr.device)
    if out.dtype != torch.int32 or out.dim() != 2 or out.shape != (nsrc, n) or (n > 1 and out.stride(1) != 1):
        raise ValueError("out must be a row-major nsrc x n int32 tensor")
    ldo = int(out.stride(0)) if nsrc > 1 else max(1, n)
    s = _stream_handle(row_ptr, stream)
    with torch.cuda.device(row_ptr.device):
        _check(lib.apsp_sssp_delta_i32(row_ptr.data_ptr(), col_idx.data_ptr(), w.data_ptr(), n,
                                       sources.data_ptr(), nsrc, int(delta), out.data_ptr(), ldo, s),
               "apsp_sssp_delta_i32")
    return out


def sssp(row_ptr, col_idx, w, source: int, delta: int = 0, out=None, stream=None):
    """One Delta-stepping search from `source` over the whole GPU on a CSR
    graph with weights >= 0 (include/apsp_sparse.h, apsp_sssp_i32).  Returns
    (or fills) an int32 CUDA tensor of n distances, INF for unreachable.
    Blocks until done."""
    import torch

    lib = load()
    n = _csr_args(row_ptr, col_idx, w)
    if out is None:
        out = torch.empty(max(n, 1), dtype=torch.int32, device=row_ptr.device)[:n]
    if out.dtype != torch.int32 or not out.is_cuda or out.dim() != 1 or out.numel() != n or not out.is_contiguous():
        raise ValueError("out must be a contiguous int32 CUDA tensor of n entries")
    s = _stream_handle(row_ptr, stream)
    with torch.cuda.device(row_ptr.device):
        _check(lib.apsp_sssp_i32(row_ptr.data_ptr(), col_idx.data_ptr() if col_idx.numel() else None,
                                 w.data_ptr() if w.numel() else None, n, int(source), int(delta),
                                 out.data_ptr(), s), "apsp_sssp_i32")
    return out


class SsspGraph:
    """A CSR graph prepared once for repeated single-source searches
    (apsp_sssp_graph_* in include/apsp_sparse.h).  The library keeps its own
    device copy, so the tensors passed in may be dropped afterwards."""

    def __init__(self, row_ptr, col_idx, w, delta: int = 0, stream=None):
        import torch

        lib = load()
        n = _csr_args(row_ptr, col_idx, w)
        self._dev = row_ptr.device
        h = ctypes.c_void_p()
        s = _stream_handle(row_ptr, stream)
        with torch.cuda.device(self._dev):
            _check(lib.apsp_sssp_graph_create(row_ptr.data_ptr(), col_idx.data_ptr() if col_idx.numel() else None,
                                              w.data_ptr() if w.numel() else None, n, int(delta), s,
                                              ctypes.byref(h)), "apsp_sssp_graph_create")
        self._h = h

    def info(self):
        """(n, m, delta)."""
        n, m, d = ctypes.c_int(), ctypes.c_longlong(), ctypes.c_int()
        _check(load().apsp_sssp_graph_info(self._h, ctypes.byref(n), ctypes.byref(m), ctypes.byref(d)),
               "apsp_sssp_graph_info")
        return n.value, m.value, d.value

    def search(self, source: int, out=None, stream=None):
        import torch

        n = self.info()[0]
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device=self._dev)
        if out.dtype != torch.int32 or out.dim() != 1 or out.numel() != n or not out.is_contiguous():
            raise ValueError("out must be a contiguous int32 CUDA tensor of n entries")
        s = _stream_handle(out, stream)
        with torch.cuda.device(self._dev):
            _check(load().apsp_sssp_graph_search(self._h, int(source), out.data_ptr(), s), "apsp_sssp_graph_search")
        return out

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _check(load().apsp_sssp_graph_destroy(self._h), "apsp_sssp_graph_destroy")
        self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def sparse_release() -> None:
    _check(load().apsp_sparse_release(), "apsp_sparse_release")


def sparse_timing_enable(enable: bool = True) -> None:
    _check(load().apsp_sparse_timing_enable(int(bool(enable))), "apsp_sparse_timing_enable")


def sparse_timing_read():
    """(search-kernel ms, search launches, sparse kernel launches) since the
    last read (include/apsp_sparse.h)."""
    ms, n, k = ctypes.c_double(), ctypes.c_longlong(), ctypes.c_longlong()
    _check(load().apsp_sparse_timing_read(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(k)),
           "apsp_sparse_timing_read")
    return ms.value, n.value, k.value


def debug_inject_grid_timeout(timeout_ns: int) -> None:
    """Test hook (include/apsp_debug.h): the next grid-wide search loses CTA 0
    before its first grid barrier, so the other CTAs' bounded waits run out
    after `timeout_ns` and the call raises ApspError(ETIMEOUT)."""
    _check(load().apsp_debug_inject_grid_timeout(int(timeout_ns)), "apsp_debug_inject_grid_timeout")
