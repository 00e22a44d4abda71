"""CPU oracle for all-pairs shortest paths -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the bench's CPU-baseline / reference leg
may import this package.  The library (min_graph_gb300) never does, and the
two share no code: this package builds its own C source (oracle.c) with gcc.

What it computes is the plain definition of the result the blocked
Floyd-Warshall method reaches (thesis page, 1library.co excerpt, section 4.6;
tiling changes no value -- "Loops into zones" page, closing paragraph):
D[i][j] = least total weight over directed paths i ~> j, INF if none, 0 on the
diagonal.  Two independent algorithms give it:

  fw_i32 / fw_f64          Floyd-Warshall triple loop (k outermost), untiled.
  dijkstra_i32 / _f32      binary-heap Dijkstra per source (Johnson/Dijkstra
                           page, CEUR Vol-1631, the sequential Dijkstra
                           operators); reverse=True gives columns.
  bfs_hops_i32             reachability / hop counts.
  bellman_ford_i32         single-source Bellman-Ford with the negative-cycle
                           check (Johnson/Dijkstra page).
  johnson_i32              Johnson's APSP as that page lays it out: negative
                           arc weights allowed, negative cycles reported.
  dijkstra_csr_i32         the same Dijkstra read from a CSR arc list (for
                           sparse graphs too large for a dense matrix).

int32 matrices use INF = 0x3FFFFFFF; floating point is computed in double
with +inf for "no arc".

Pins (tests/test_oracle_pins.py): hand-worked graphs under tests/golden/,
brute-force enumeration of simple paths for n <= 7, closed forms (directed
path, metric on a line, unit weights = BFS hops), invariants, FW == Dijkstra,
and planted mistakes that the pins must catch.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

INF_I32 = 0x3FFFFFFF

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> None:
    """gcc -O2 with OpenMP when the toolchain has it, else without."""
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", out, "-lm"]
    try:
        subprocess.check_call(base[:1] + ["-fopenmp"] + base[1:], stderr=subprocess.DEVNULL)
    except subprocess.CalledProcessError:
        subprocess.check_call(base)


def build(force: bool = False) -> str:
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(SOURCE):
        tmp = _SO + f".tmp{os.getpid()}"
        compile_source(SOURCE, tmp)
        os.replace(tmp, _SO)
    return _SO


def bind(path: str):
    """Load an oracle shared object and declare its signatures."""
    lib = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_has_openmp.argtypes = []
    lib.oracle_has_openmp.restype = i32
    lib.oracle_fw_i32.argtypes = [vp, i64, i64, i32]
    lib.oracle_fw_i32.restype = i32
    lib.oracle_fw_i32_steps.argtypes = [vp, i64, i64, i64, i64, i32]
    lib.oracle_fw_i32_steps.restype = i32
    lib.oracle_fw_f64.argtypes = [vp, i64, i64, i32]
    lib.oracle_fw_f64.restype = i32
    lib.oracle_fw_f64_steps.argtypes = [vp, i64, i64, i64, i64, i32]
    lib.oracle_fw_f64_steps.restype = i32
    lib.oracle_dijkstra_i32.argtypes = [vp, i64, i64, vp, i64, i32, vp, i32]
    lib.oracle_dijkstra_i32.restype = i32
    lib.oracle_dijkstra_f32.argtypes = [vp, i64, i64, vp, i64, i32, vp, i32]
    lib.oracle_dijkstra_f32.restype = i32
    lib.oracle_bfs_hops_i32.argtypes = [vp, i64, i64, i64, vp]
    lib.oracle_bfs_hops_i32.restype = i32
    lib.oracle_bellman_ford_i32.argtypes = [vp, i64, i64, i64, vp]
    lib.oracle_bellman_ford_i32.restype = i32
    lib.oracle_johnson_i32.argtypes = [vp, i64, i64, vp, i32]
    lib.oracle_johnson_i32.restype = i32
    lib.oracle_johnson_rows_i32.argtypes = [vp, i64, i64, vp, i64, vp, i32]
    lib.oracle_johnson_rows_i32.restype = i32
    lib.oracle_dijkstra_csr_i32.argtypes = [vp, vp, vp, i64, vp, i64, vp, i32]
    lib.oracle_dijkstra_csr_i32.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def has_openmp() -> bool:
    return bool(_load().oracle_has_openmp())


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _as_matrix(w: np.ndarray, dtype) -> np.ndarray:
    w = np.asarray(w)
    if w.ndim != 2 or w.dtype != dtype:
        raise TypeError(f"expected a 2-D {np.dtype(dtype)} matrix")
    if not w.flags.c_contiguous:
        w = np.ascontiguousarray(w)
    return w


class Oracle:
    """The oracle bound to one shared object (the built one by default; the
    pin tests also bind deliberately broken builds to show the pins fail)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else _load()

    def fw_i32(self, w: np.ndarray, n: int | None = None, threads: int = 1) -> np.ndarray:
        """Floyd-Warshall on a copy of an int32 matrix (n x ld, ld >= n).
        Returns the n x n distance matrix (INF = 0x3FFFFFFF)."""
        w = _as_matrix(w, np.int32)
        n = w.shape[0] if n is None else n
        d = np.array(w[:n, :n], dtype=np.int32, order="C", copy=True)
        _check(self.lib.oracle_fw_i32(d.ctypes.data, n, n, threads), "fw_i32")
        return d

    def fw_i32_steps(self, d: np.ndarray, k_begin: int, k_end: int, threads: int = 1) -> None:
        """Floyd-Warshall steps k_begin..k_end-1 in place (bounded samples)."""
        d = _as_matrix(d, np.int32)
        n = d.shape[0]
        _check(self.lib.oracle_fw_i32_steps(d.ctypes.data, n, d.shape[1], k_begin, k_end, threads),
               "fw_i32_steps")

    def fw_f64(self, w: np.ndarray, n: int | None = None, threads: int = 1) -> np.ndarray:
        """Floyd-Warshall in double on a float32/float64 matrix; +inf = no path."""
        w = np.asarray(w)
        n = w.shape[0] if n is None else n
        d = np.array(w[:n, :n], dtype=np.float64, order="C", copy=True)
        _check(self.lib.oracle_fw_f64(d.ctypes.data, n, n, threads), "fw_f64")
        return d

    def fw_f64_steps(self, d: np.ndarray, k_begin: int, k_end: int, threads: int = 1) -> None:
        """Floyd-Warshall steps k_begin..k_end-1 in place on a float64 matrix."""
        d = _as_matrix(d, np.float64)
        _check(self.lib.oracle_fw_f64_steps(d.ctypes.data, d.shape[0], d.shape[1], k_begin, k_end, threads),
               "fw_f64_steps")

    def dijkstra_i32(self, w: np.ndarray, sources, reverse: bool = False,
                     threads: int | None = None, n: int | None = None) -> np.ndarray:
        """Rows D[s, :] (or columns D[:, s] with reverse) for an int32 matrix."""
        w = _as_matrix(w, np.int32)
        n = w.shape[0] if n is None else n
        src = np.ascontiguousarray(np.asarray(sources, dtype=np.int32))
        out = np.empty((src.size, n), dtype=np.int32)
        _check(self.lib.oracle_dijkstra_i32(w.ctypes.data, n, w.shape[1], src.ctypes.data, src.size,
                                            int(reverse), out.ctypes.data,
                                            threads or default_threads()), "dijkstra_i32")
        return out

    def dijkstra_f32(self, w: np.ndarray, sources, reverse: bool = False,
                     threads: int | None = None, n: int | None = None) -> np.ndarray:
        """Rows (or columns) for an fp32 matrix, accumulated in double."""
        w = _as_matrix(w, np.float32)
        n = w.shape[0] if n is None else n
        src = np.ascontiguousarray(np.asarray(sources, dtype=np.int32))
        out = np.empty((src.size, n), dtype=np.float64)
        _check(self.lib.oracle_dijkstra_f32(w.ctypes.data, n, w.shape[1], src.ctypes.data, src.size,
                                            int(reverse), out.ctypes.data,
                                            threads or default_threads()), "dijkstra_f32")
        return out

    def bellman_ford_i32(self, w: np.ndarray, src: int):
        """Distances from src (int64, INF = 0x3FFFFFFF for unreachable), or
        None when a negative cycle is reachable from src."""
        w = _as_matrix(w, np.int32)
        out = np.empty(w.shape[0], dtype=np.int64)
        rc = self.lib.oracle_bellman_ford_i32(w.ctypes.data, w.shape[0], w.shape[1], src, out.ctypes.data)
        if rc == 1:
            return None
        _check(rc, "bellman_ford_i32")
        return out

    def johnson_i32(self, w: np.ndarray, threads: int | None = None):
        """All-pairs distances by Johnson's method (negative arc weights
        allowed), int32 with INF; None when the graph has a negative cycle."""
        w = _as_matrix(w, np.int32)
        n = w.shape[0]
        out = np.empty((n, n), dtype=np.int32)
        rc = self.lib.oracle_johnson_i32(w.ctypes.data, n, w.shape[1], out.ctypes.data,
                                         threads or default_threads())
        if rc == 1:
            return None
        _check(rc, "johnson_i32")
        return out

    def dijkstra_csr_i32(self, row_ptr: np.ndarray, col: np.ndarray, w: np.ndarray, sources,
                         threads: int | None = None) -> np.ndarray:
        """Rows of distances from `sources` on a CSR graph (int64 row_ptr,
        int32 col and w >= 0); int32 with INF for unreachable."""
        row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
        col = np.ascontiguousarray(col, dtype=np.int32)
        w = np.ascontiguousarray(w, dtype=np.int32)
        n = row_ptr.size - 1
        src = np.ascontiguousarray(np.asarray(sources, dtype=np.int32))
        out = np.empty((src.size, n), dtype=np.int32)
        _check(self.lib.oracle_dijkstra_csr_i32(row_ptr.ctypes.data, col.ctypes.data, w.ctypes.data, n,
                                                src.ctypes.data, src.size, out.ctypes.data,
                                                threads or default_threads()), "dijkstra_csr_i32")
        return out

    def johnson_rows_i32(self, w: np.ndarray, sources, threads: int | None = None):
        """Rows of Johnson's all-pairs distances for the given sources only
        (the potentials still come from Bellman-Ford over the whole graph);
        None on a negative cycle."""
        w = _as_matrix(w, np.int32)
        n = w.shape[0]
        src = np.ascontiguousarray(np.asarray(sources, dtype=np.int32))
        out = np.empty((src.size, n), dtype=np.int32)
        rc = self.lib.oracle_johnson_rows_i32(w.ctypes.data, n, w.shape[1], src.ctypes.data, src.size,
                                              out.ctypes.data, threads or default_threads())
        if rc == 1:
            return None
        _check(rc, "johnson_rows_i32")
        return out

    def bfs_hops_i32(self, w: np.ndarray, src: int) -> np.ndarray:
        w = _as_matrix(w, np.int32)
        hops = np.empty(w.shape[0], dtype=np.int32)
        _check(self.lib.oracle_bfs_hops_i32(w.ctypes.data, w.shape[0], w.shape[1], src,
                                            hops.ctypes.data), "bfs_hops_i32")
        return hops


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def fw_i32(w, threads: int = 1):
    return default().fw_i32(w, threads=threads)


def fw_f64(w, threads: int = 1):
    return default().fw_f64(w, threads=threads)


def dijkstra_i32(w, sources, reverse=False, threads=None):
    return default().dijkstra_i32(w, sources, reverse=reverse, threads=threads)


def dijkstra_f32(w, sources, reverse=False, threads=None):
    return default().dijkstra_f32(w, sources, reverse=reverse, threads=threads)


def bfs_hops_i32(w, src):
    return default().bfs_hops_i32(w, src)


def bellman_ford_i32(w, src):
    return default().bellman_ford_i32(w, src)


def johnson_i32(w, threads=None):
    return default().johnson_i32(w, threads=threads)


def dijkstra_csr_i32(row_ptr, col, w, sources, threads=None):
    return default().dijkstra_csr_i32(row_ptr, col, w, sources, threads=threads)


def johnson_rows_i32(w, sources, threads=None):
    return default().johnson_rows_i32(w, sources, threads=threads)
