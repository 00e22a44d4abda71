"""Seeded synthetic graph inputs (dense distance matrices), shared by the
tests, the bench and the oracle's pins.

This module holds no shortest-path arithmetic.  It draws directed
Erdos-Renyi and Barabasi-Albert graphs as dense row-major matrices with INF
where there is no arc and 0 on the diagonal, which is the problem statement
of the blocked Floyd-Warshall thesis page (1library.co excerpt, section 4.6:
the whole graph held as a matrix in global memory).  The C side (gen.c) is
built with gcc on first use; the same source gives the same matrices on x86
and Arm.

The five standard workloads:

  er256   : directed ER, n=256,   p=0.1,  int32 w in [1,100],   seed 1
  er2048  : directed ER, n=2048,  p=0.05, int32 w in [1,1000],  seed 2
  er8192  : directed ER, n=8192,  p=0.5,  int32 w in [1,10000], seed 3
  ba16384 : Barabasi-Albert beta=8, 2 arcs per edge, n=16384,
            int32 w in [1,1000], seed 4
  er32768 : directed ER, n=32768, p=0.01, fp32 w in (0,1], seed 5
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

INF_I32 = 0x3FFFFFFF
INF_F32 = np.float32(np.inf)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libgraphgen.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into _build/libgraphgen.so (gcc, portable flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u64, i32, dbl, vp = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.graphgen_splitmix64_at.argtypes = [u64, u64]
            lib.graphgen_splitmix64_at.restype = u64
            lib.graphgen_er_i32.argtypes = [vp, i64, i64, i64, i64, dbl, i32, i32, i32, u64]
            lib.graphgen_er_i32.restype = None
            lib.graphgen_er_f32.argtypes = [vp, i64, i64, i64, i64, dbl, u64]
            lib.graphgen_er_f32.restype = None
            lib.graphgen_er_potential_i32.argtypes = [vp, i64, i64, i64, i64, dbl, i32, i32, i32, i32, u64]
            lib.graphgen_er_potential_i32.restype = None
            lib.graphgen_ba_edges.argtypes = [vp, i64, i32, u64]
            lib.graphgen_ba_edges.restype = i64
            lib.graphgen_ba_i32.argtypes = [vp, i64, i64, i32, i32, i32, i32, u64]
            lib.graphgen_ba_i32.restype = i64
            lib.graphgen_rmat_arcs.argtypes = [vp, vp, vp, i64, i64, i32, dbl, dbl, dbl, i32, i32, u64]
            lib.graphgen_rmat_arcs.restype = None
            lib.graphgen_csr_from_arcs.argtypes = [vp, vp, vp, i64, i64, vp, vp, vp]
            lib.graphgen_csr_from_arcs.restype = i32
            _lib = lib
    return _lib


def splitmix64_at(seed: int, t: int) -> int:
    """t-th output (t >= 1) of SplitMix64 seeded with `seed`."""
    return int(_load().graphgen_splitmix64_at(seed & (2**64 - 1), t))


def _alloc(n: int, ld: int | None, dtype, out):
    ld = n if ld is None else ld
    if ld < n:
        raise ValueError("ld < n")
    if out is None:
        out = np.empty((n, ld), dtype=dtype)
    if out.shape != (n, ld) or out.dtype != dtype or not out.flags.c_contiguous:
        raise ValueError("out must be a C-contiguous (n, ld) array of the right dtype")
    return out, ld


def _rows_parallel(fn, n: int, threads: int | None):
    threads = threads or min(16, os.cpu_count() or 1)
    chunk = max(64, (n + threads * 4 - 1) // (threads * 4))
    spans = [(b, min(n, b + chunk)) for b in range(0, n, chunk)]
    if len(spans) <= 1:
        for b, e in spans:
            fn(b, e)
        return
    with ThreadPoolExecutor(max_workers=threads) as ex:  # ctypes releases the GIL
        list(ex.map(lambda s: fn(*s), spans))


def er_i32(n: int, p: float, wlo: int, whi: int, seed: int, ld: int | None = None,
           out: np.ndarray | None = None, inf: int = INF_I32, threads: int | None = None) -> np.ndarray:
    """Directed Erdos-Renyi G(n, p), int32 weights uniform in [wlo, whi]."""
    out, ld = _alloc(n, ld, np.int32, out)
    lib = _load()
    base = out.ctypes.data

    def rows(b, e):
        lib.graphgen_er_i32(base + b * ld * 4, n, ld, b, e, p, wlo, whi, inf, seed)

    _rows_parallel(rows, n, threads)
    return out


def er_f32(n: int, p: float, seed: int, ld: int | None = None, out: np.ndarray | None = None,
           threads: int | None = None) -> np.ndarray:
    """Directed Erdos-Renyi G(n, p), fp32 weights in (0, 1] on a 2^-24 grid, +inf for no arc."""
    out, ld = _alloc(n, ld, np.float32, out)
    lib = _load()
    base = out.ctypes.data

    def rows(b, e):
        lib.graphgen_er_f32(base + b * ld * 4, n, ld, b, e, p, seed)

    _rows_parallel(rows, n, threads)
    return out


def er_potential_i32(n: int, p: float, wlo: int, whi: int, pmax: int, seed: int,
                     ld: int | None = None, out: np.ndarray | None = None, inf: int = INF_I32,
                     threads: int | None = None) -> np.ndarray:
    """Directed ER graph with negative arc weights but no negative cycle:
    w(i, j) = w0(i, j) + p(i) - p(j), w0 uniform in [wlo, whi] (wlo >= 0),
    vertex potentials p uniform in [0, pmax]."""
    if wlo < 0:
        raise ValueError("wlo must be >= 0")
    out, ld = _alloc(n, ld, np.int32, out)
    lib = _load()
    base = out.ctypes.data

    def rows(b, e):
        lib.graphgen_er_potential_i32(base + b * ld * 4, n, ld, b, e, p, wlo, whi, pmax, inf, seed)

    _rows_parallel(rows, n, threads)
    return out


def ba_edges(n: int, beta: int, seed: int) -> np.ndarray:
    """Barabasi-Albert undirected edge list, shape (beta*(n-beta), 2)."""
    m = beta * (n - beta)
    edges = np.empty((m, 2), dtype=np.int32)
    got = _load().graphgen_ba_edges(edges.ctypes.data, n, beta, seed)
    if got != m:
        raise ValueError("bad Barabasi-Albert arguments")
    return edges


def ba_i32(n: int, beta: int, wlo: int, whi: int, seed: int, ld: int | None = None,
           out: np.ndarray | None = None, inf: int = INF_I32) -> np.ndarray:
    """Barabasi-Albert graph as a dense int32 matrix, two arcs per edge."""
    out, ld = _alloc(n, ld, np.int32, out)
    arcs = _load().graphgen_ba_i32(out.ctypes.data, n, ld, beta, wlo, whi, inf, seed)
    if arcs != 2 * beta * (n - beta):
        raise ValueError("bad Barabasi-Albert arguments")
    return out


RMAT_ABC = (0.57, 0.19, 0.19)  # Graph500 quadrant probabilities (d = 0.05)


def rmat_csr(scale: int, edge_factor: int = 32, wlo: int = 1, whi: int = 1 << 20, seed: int = 6,
             abc=RMAT_ABC, threads: int | None = None):
    """R-MAT graph with 2^scale vertices and edge_factor * 2^scale arcs, as
    CSR (row_ptr int64[n+1], col int32[m], w int32[m]); see gen.c for the
    recipe (Graph500 quadrant probabilities, scrambled vertex ids, int32
    weights uniform in [wlo, whi], self-loops and parallel arcs kept)."""
    if not 1 <= scale <= 30:
        raise ValueError("scale must be in [1, 30]")
    n = 1 << scale
    m = edge_factor * n
    tail = np.empty(m, dtype=np.int32)
    head = np.empty(m, dtype=np.int32)
    wt = np.empty(m, dtype=np.int32)
    lib = _load()
    a, b, c = abc

    def arcs(e0, e1):
        lib.graphgen_rmat_arcs(tail.ctypes.data + 4 * e0, head.ctypes.data + 4 * e0, wt.ctypes.data + 4 * e0,
                               e0, e1, scale, a, b, c, wlo, whi, seed)

    _rows_parallel(arcs, m, threads)
    row_ptr = np.empty(n + 1, dtype=np.int64)
    col = np.empty(m, dtype=np.int32)
    w = np.empty(m, dtype=np.int32)
    rc = lib.graphgen_csr_from_arcs(tail.ctypes.data, head.ctypes.data, wt.ctypes.data, m, n,
                                    row_ptr.ctypes.data, col.ctypes.data, w.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"graphgen_csr_from_arcs failed: {rc}")
    return row_ptr, col, w


def describe_rmat(scale: int, edge_factor: int = 32, wlo: int = 1, whi: int = 1 << 20, seed: int = 6) -> str:
    return (f"R-MAT scale {scale} (n = {1 << scale}), {edge_factor} arcs per vertex, "
            f"(a,b,c,d) = (0.57,0.19,0.19,0.05), int32 w in [{wlo},{whi}], seed {seed}")


# name -> (kind, n, params, dtype)
CONFIGS = {
    "er256": dict(kind="er", n=256, p=0.1, wlo=1, whi=100, seed=1, dtype="int32"),
    "er2048": dict(kind="er", n=2048, p=0.05, wlo=1, whi=1000, seed=2, dtype="int32"),
    "er8192": dict(kind="er", n=8192, p=0.5, wlo=1, whi=10000, seed=3, dtype="int32"),
    "ba16384": dict(kind="ba", n=16384, beta=8, wlo=1, whi=1000, seed=4, dtype="int32"),
    "er32768": dict(kind="er", n=32768, p=0.01, seed=5, dtype="float32"),
}


def make(name: str, ld: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Build one of the five standard workloads as a host matrix."""
    c = CONFIGS[name]
    if c["kind"] == "ba":
        return ba_i32(c["n"], c["beta"], c["wlo"], c["whi"], c["seed"], ld=ld, out=out)
    if c["dtype"] == "float32":
        return er_f32(c["n"], c["p"], c["seed"], ld=ld, out=out)
    return er_i32(c["n"], c["p"], c["wlo"], c["whi"], c["seed"], ld=ld, out=out)


def describe(name: str) -> str:
    c = CONFIGS[name]
    if c["kind"] == "ba":
        return (f"Barabasi-Albert beta={c['beta']} (2 arcs per edge), n={c['n']}, "
                f"int32 w in [{c['wlo']},{c['whi']}], seed {c['seed']}")
    if c["dtype"] == "float32":
        return f"directed ER n={c['n']} p={c['p']}, fp32 w in (0,1], seed {c['seed']}"
    return (f"directed ER n={c['n']} p={c['p']}, int32 w in [{c['wlo']},{c['whi']}], "
            f"seed {c['seed']}")
