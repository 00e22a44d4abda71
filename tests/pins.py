"""Checks that pin the CPU oracle to facts other than itself.

Every check returns a list of failure strings (empty = pass), so the same
checks run against the real oracle (tests/test_oracle_pins.py) and against
deliberately broken builds of it (the planted-mistake test), where at least
one of them must fail.

None of these re-types the oracle's recurrence: they use hand-worked values
(tests/golden/), brute-force enumeration of simple paths, closed forms,
breadth-first search written here, and invariants of shortest paths.
"""
from __future__ import annotations

import glob
import os
from collections import deque

import numpy as np

import graphgen

INF = 0x3FFFFFFF
GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- golden files

def golden_flags(path: str) -> set:
    """Flag lines of a fixture: 'negative' (negative arc weights, Dijkstra does
    not apply), 'negative_cycle' (no distances exist; no D section)."""
    flags = set()
    with open(path) as f:
        for line in f:
            if line.strip() in ("negative", "negative_cycle"):
                flags.add(line.strip())
    return flags


def load_golden(path: str):
    """Parse a golden fixture: returns (name, dtype, W, D); D is None for a
    negative-cycle fixture."""
    dtype, n, mode, rows = None, None, None, {"W": [], "D": []}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#") or line in ("negative", "negative_cycle"):
                continue
            if line.startswith("dtype"):
                dtype = line.split()[1]
            elif line.startswith("n "):
                n = int(line.split()[1])
            elif line in ("W", "D"):
                mode = line
            else:
                rows[mode].append(line.split())
    assert dtype in ("int32", "float32") and n is not None

    def conv(tok):
        if dtype == "int32":
            return INF if tok == "INF" else int(tok)
        return float(tok)

    w = np.array([[conv(t) for t in r] for r in rows["W"]],
                 dtype=np.int64 if dtype == "int32" else np.float32)
    d = None
    if rows["D"]:
        d = np.array([[conv(t) for t in r] for r in rows["D"]],
                     dtype=np.int64 if dtype == "int32" else np.float64)
        assert d.shape == (n, n)
    assert w.shape == (n, n)
    if dtype == "int32":
        w = np.minimum(w, 2**31 - 1).astype(np.int32)
    return os.path.basename(path), dtype, w, d


def golden_files():
    return sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt")))


def check_golden(orc) -> list[str]:
    bad = []
    for path in golden_files():
        name, dtype, w, d = load_golden(path)
        n = w.shape[0]
        flags = golden_flags(path)
        if "negative_cycle" in flags:
            if orc.johnson_i32(w) is not None:
                bad.append(f"golden {name}: Johnson missed the negative cycle")
            if any(orc.bellman_ford_i32(w, s) is not None for s in range(n)):
                bad.append(f"golden {name}: Bellman-Ford missed the negative cycle")
            continue
        if "negative" in flags:
            outs = {"fw": orc.fw_i32(w), "johnson": orc.johnson_i32(w, threads=1)}
            outs["bellman-ford"] = np.stack([orc.bellman_ford_i32(w, s) for s in range(n)])
            for k, got in outs.items():
                if got is None or not np.array_equal(np.asarray(got).astype(np.int64), d):
                    bad.append(f"golden {name}: {k} differs")
            continue
        if dtype == "int32":
            outs = {"fw": orc.fw_i32(w), "dijkstra": orc.dijkstra_i32(w, np.arange(n), threads=1),
                    "dijkstra-cols": orc.dijkstra_i32(w, np.arange(n), reverse=True, threads=1).T}
            for k, got in outs.items():
                if not np.array_equal(got.astype(np.int64), d):
                    bad.append(f"golden {name}: {k} differs")
        else:
            outs = {"fw": orc.fw_f64(w), "dijkstra": orc.dijkstra_f32(w, np.arange(n), threads=1)}
            for k, got in outs.items():
                if not np.array_equal(got, d):
                    bad.append(f"golden {name}: {k} differs")
    return bad


# ---------------------------------------------------------------- brute force

def brute_force(w: np.ndarray, integer: bool) -> np.ndarray:
    """Least weight over all simple directed paths, by depth-first enumeration.
    A shortest path with non-negative weights can always be taken simple."""
    n = w.shape[0]
    noarc = (lambda x: x >= INF) if integer else (lambda x: np.isinf(x))
    best = np.full((n, n), np.inf)
    for s in range(n):
        best[s, s] = 0.0
        stack = [(s, 0.0, 1 << s)]
        while stack:
            u, dist, seen = stack.pop()
            for v in range(n):
                if v == u or (seen >> v) & 1 or noarc(w[u, v]):
                    continue
                nd = dist + float(w[u, v])
                if nd < best[s, v]:
                    best[s, v] = nd
                stack.append((v, nd, seen | (1 << v)))
    if integer:
        out = np.where(best >= INF, INF, best)
        return out.astype(np.int64)
    return best


def random_small(seed: int, integer: bool):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 8))
    p = float(rng.choice([0.15, 0.4, 0.8]))
    if integer:
        w = graphgen.er_i32(n, p, 0, 9, seed) if seed % 3 else graphgen.er_i32(n, p, 1, 100, seed)
    else:
        w = graphgen.er_f32(n, p, seed)
    return w


def check_brute_force(orc, seeds=range(60)) -> list[str]:
    bad = []
    for seed in seeds:
        w = random_small(seed, True)
        n = w.shape[0]
        ref = brute_force(w, True)
        for k, got in (("fw", orc.fw_i32(w)), ("dijkstra", orc.dijkstra_i32(w, np.arange(n), threads=1))):
            if not np.array_equal(got.astype(np.int64), ref):
                bad.append(f"brute force int seed {seed}: {k} differs")
        wf = random_small(seed, False)
        n = wf.shape[0]
        ref = brute_force(wf, False)
        for k, got in (("fw", orc.fw_f64(wf)), ("dijkstra", orc.dijkstra_f32(wf, np.arange(n), threads=1))):
            fin = np.isfinite(ref)
            if not (np.array_equal(np.isfinite(got), fin)
                    and np.allclose(got[fin], ref[fin], rtol=1e-12, atol=0)):
                bad.append(f"brute force f64 seed {seed}: {k} differs")
    return bad


# ---------------------------------------------------------------- closed forms

def check_closed_forms(orc) -> list[str]:
    bad = []
    rng = np.random.default_rng(1234)
    # Directed path 0->1->...->n-1: D[i][j] = w_i + ... + w_{j-1} for i <= j,
    # INF for i > j.  n = 300 is not a multiple of any tile size.
    n = 300
    wts = rng.integers(0, 1000, size=n - 1)
    w = np.full((n, n), INF, dtype=np.int32)
    np.fill_diagonal(w, 0)
    w[np.arange(n - 1), np.arange(1, n)] = wts
    pref = np.concatenate([[0], np.cumsum(wts)])
    ref = np.where(np.arange(n)[:, None] <= np.arange(n)[None, :],
                   pref[None, :] - pref[:, None], INF)
    if not np.array_equal(orc.fw_i32(w).astype(np.int64), ref):
        bad.append("closed form: directed path (fw)")
    if not np.array_equal(orc.dijkstra_i32(w, np.arange(n), threads=1).astype(np.int64), ref):
        bad.append("closed form: directed path (dijkstra)")
    # Complete graph of points on a line, W[i][j] = |x_i - x_j|: the metric
    # already satisfies the triangle inequality, so D = W.
    n = 97
    x = rng.integers(0, 10**6, size=n)
    w = np.abs(x[:, None] - x[None, :]).astype(np.int32)
    if not np.array_equal(orc.fw_i32(w), w):
        bad.append("closed form: line metric (fw)")
    if not np.array_equal(orc.dijkstra_i32(w, np.arange(n), threads=1), w):
        bad.append("closed form: line metric (dijkstra)")
    # Same in floating point with dyadic coordinates (exact sums).
    xf = rng.integers(0, 2**20, size=n) / 1024.0
    wf = np.abs(xf[:, None] - xf[None, :]).astype(np.float32)
    if not np.array_equal(orc.fw_f64(wf), wf.astype(np.float64)):
        bad.append("closed form: line metric (fw_f64)")
    # Unit weights: D = breadth-first hop count (BFS written here).
    for seed in (11, 12, 13):
        w = graphgen.er_i32(150, 0.02 * (seed - 10), 1, 1, seed)
        hops = bfs_all(w)
        if not np.array_equal(orc.fw_i32(w).astype(np.int64), hops):
            bad.append(f"closed form: unit weights vs BFS seed {seed} (fw)")
        if not np.array_equal(orc.dijkstra_i32(w, np.arange(150), threads=1).astype(np.int64), hops):
            bad.append(f"closed form: unit weights vs BFS seed {seed} (dijkstra)")
        # The oracle's own BFS (-1 where unreachable) against the one here.
        for src in (0, 37, 149):
            got = orc.bfs_hops_i32(w, src).astype(np.int64)
            got[got < 0] = INF
            if not np.array_equal(got, hops[src]):
                bad.append(f"closed form: oracle BFS hops vs BFS seed {seed} source {src}")
    return bad


def bfs_all(w: np.ndarray) -> np.ndarray:
    """Hop counts from every source (INF where unreachable), by BFS."""
    n = w.shape[0]
    adj = [np.nonzero((w[u] < INF) & (np.arange(n) != u))[0] for u in range(n)]
    out = np.full((n, n), INF, dtype=np.int64)
    for s in range(n):
        out[s, s] = 0
        q = deque([s])
        while q:
            u = q.popleft()
            for v in adj[u]:
                if out[s, v] == INF:
                    out[s, v] = out[s, u] + 1
                    q.append(v)
    return out


# ---------------------------------------------------------------- invariants

def invariant_failures_i32(w: np.ndarray, d: np.ndarray, reach: np.ndarray | None = None) -> list[str]:
    """Properties every correct int32 APSP result has (full matrix, O(n^3))."""
    bad = []
    n = w.shape[0]
    d = d.astype(np.int64)
    wc = np.minimum(w.astype(np.int64), INF)
    if not np.all(np.diag(d) == 0):
        bad.append("D[i,i] != 0")
    if np.any(d > wc):
        bad.append("D > W somewhere")
    for k in range(n):  # triangle inequality, saturating at INF
        via = np.minimum(d[:, k][:, None] + d[k, :][None, :], INF)
        if np.any(d > via):
            bad.append(f"triangle inequality fails through k={k}")
            break
    if reach is not None and not np.array_equal(d < INF, reach):
        bad.append("INF pattern differs from reachability")
    # every finite D[i,j], i != j, is realised by a first arc i->k
    fin = (d < INF) & ~np.eye(n, dtype=bool)
    arc = (wc < INF) & ~np.eye(n, dtype=bool)
    realised = np.zeros((n, n), dtype=bool)
    for k in range(n):
        ok = arc[:, k][:, None] & (wc[:, k][:, None] + d[k, :][None, :] == d)
        realised |= ok
    if np.any(fin & ~realised):
        bad.append("a finite distance is not realised by any first arc")
    return bad


def check_invariants(orc) -> list[str]:
    bad = []
    for seed, (n, p) in enumerate([(120, 0.02), (160, 0.05), (200, 0.3), (64, 0.0)]):
        w = graphgen.er_i32(n, p, 1, 1000, 100 + seed)
        d = orc.fw_i32(w)
        reach = bfs_all(w) < INF
        bad += [f"invariants seed {seed}: {m}" for m in invariant_failures_i32(w, d, reach)]
    w = graphgen.ba_i32(300, 3, 1, 1000, 77)
    d = orc.fw_i32(w)
    bad += [f"invariants BA: {m}" for m in invariant_failures_i32(w, d, bfs_all(w) < INF)]
    return bad


# ---------------------------------------------------------------- agreement

def check_fw_vs_dijkstra(orc) -> list[str]:
    bad = []
    for seed, (n, p) in enumerate([(257, 0.01), (300, 0.05), (129, 0.5), (200, 0.003)]):
        w = graphgen.er_i32(n, p, 1, 1000, 200 + seed)
        fw = orc.fw_i32(w)
        if not np.array_equal(fw, orc.dijkstra_i32(w, np.arange(n), threads=2)):
            bad.append(f"fw != dijkstra rows, int seed {seed}")
        if not np.array_equal(fw, orc.dijkstra_i32(w, np.arange(n), reverse=True, threads=2).T):
            bad.append(f"fw != dijkstra columns, int seed {seed}")
        wf = graphgen.er_f32(n, p, 300 + seed)
        ff = orc.fw_f64(wf)
        fd = orc.dijkstra_f32(wf, np.arange(n), threads=2)
        fin = np.isfinite(ff)
        if not (np.array_equal(fin, np.isfinite(fd)) and np.allclose(ff[fin], fd[fin], rtol=1e-12, atol=0)):
            bad.append(f"fw_f64 != dijkstra_f32, seed {seed}")
    return bad


def check_negative_weights(orc) -> list[str]:
    """Negative arc weights without negative cycles: brute force over simple
    paths (still the definition then), Floyd-Warshall, Johnson and
    Bellman-Ford rows must all agree; a planted negative cycle is reported."""
    bad = []
    for seed in range(40):
        rng = np.random.default_rng(500 + seed)
        n = int(rng.integers(2, 8))
        w = graphgen.er_potential_i32(n, float(rng.choice([0.3, 0.7])), 0, 20, 30, 500 + seed)
        ref = brute_force(w, True)
        jo = orc.johnson_i32(w, threads=1)
        if jo is None or not np.array_equal(jo.astype(np.int64), ref):
            bad.append(f"negative weights brute force seed {seed}: johnson differs")
        if not np.array_equal(orc.fw_i32(w).astype(np.int64), ref):
            bad.append(f"negative weights brute force seed {seed}: fw differs")
        bf = np.stack([orc.bellman_ford_i32(w, s) for s in range(n)])
        if not np.array_equal(bf, ref):
            bad.append(f"negative weights brute force seed {seed}: bellman-ford differs")
    for seed, (n, p) in enumerate([(150, 0.03), (200, 0.1), (64, 0.5)]):
        w = graphgen.er_potential_i32(n, p, 0, 100, 400, 600 + seed)
        fw = orc.fw_i32(w)
        jo = orc.johnson_i32(w, threads=2)
        if jo is None or not np.array_equal(fw, jo):
            bad.append(f"negative weights seed {seed}: johnson != fw")
        for s in (0, n // 2, n - 1):
            bfr = orc.bellman_ford_i32(w, s)
            if bfr is None or not np.array_equal(bfr, fw[s].astype(np.int64)):
                bad.append(f"negative weights seed {seed}: bellman-ford row {s} != fw")
        # plant a negative cycle: close a path with a very negative arc
        w2 = w.copy()
        w2[1, 2] = 0
        w2[2, 1] = -1
        if orc.johnson_i32(w2, threads=2) is not None:
            bad.append(f"negative weights seed {seed}: planted negative cycle not reported")
        if orc.bellman_ford_i32(w2, 1) is not None:
            bad.append(f"negative weights seed {seed}: bellman-ford missed the planted cycle")
    return bad


def random_multigraph(seed: int):
    """A small CSR multigraph: parallel arcs (up to three per ordered pair)
    and self-loops, weights in [0, 30]."""
    rng = np.random.default_rng(10_000 + seed)
    n = int(rng.integers(1, 8))
    m = int(rng.integers(0, 4 * n * n + 1))
    tail = rng.integers(0, n, m)
    head = rng.integers(0, n, m)
    wt = rng.integers(0, 31, m).astype(np.int32)
    order = np.argsort(tail, kind="stable")
    row_ptr = np.concatenate([[0], np.cumsum(np.bincount(tail, minlength=n))]).astype(np.int64)
    return n, row_ptr, head[order].astype(np.int32), wt[order], tail[order]


def check_dijkstra_csr(orc) -> list[str]:
    """The CSR Dijkstra on multigraphs against brute force over simple paths
    (parallel arcs reduce to their lightest, self-loops never help), against
    the dense Dijkstra on the same graphs, and the directed-path closed form."""
    bad = []
    for seed in range(40):
        n, row_ptr, col, wt, tail = random_multigraph(seed)
        dense = np.full((n, n), INF, dtype=np.int64)
        np.fill_diagonal(dense, 0)
        off = tail != col
        np.minimum.at(dense, (tail[off], col[off]), wt[off])
        dense = dense.astype(np.int32)
        ref = brute_force(dense, integer=True)
        got = orc.dijkstra_csr_i32(row_ptr, col, wt, np.arange(n))
        if not np.array_equal(got.astype(np.int64), ref):
            bad.append(f"dijkstra_csr seed {seed}: differs from brute force")
        if not np.array_equal(got, orc.dijkstra_i32(dense, np.arange(n))):
            bad.append(f"dijkstra_csr seed {seed}: differs from the dense Dijkstra")
    n = 50  # directed path 0 -> 1 -> ... -> 49: prefix sums
    wts = np.arange(1, n, dtype=np.int32) * 3
    row_ptr = np.concatenate([np.arange(n, dtype=np.int64), [n - 1]])
    got = orc.dijkstra_csr_i32(row_ptr, np.arange(1, n, dtype=np.int32), wts, [0, 10])
    pref = np.concatenate([[0], np.cumsum(wts)])
    if not (np.array_equal(got[0], pref) and np.array_equal(got[1, 10:], pref[10:] - pref[10])
            and np.all(got[1, :10] == INF)):
        bad.append("dijkstra_csr: directed path closed form")
    return bad


def check_johnson_rows(orc) -> list[str]:
    """Johnson's rows for chosen sources equal those rows of the full Johnson
    matrix, and of the Floyd-Warshall matrix, on negative-weight graphs."""
    bad = []
    for seed in range(6):
        n = 30 + 25 * seed
        w = graphgen.er_potential_i32(n, 0.15, 0, 200, 150, seed=700 + seed)
        src = np.random.default_rng(seed).choice(n, 5, replace=False)
        rows = orc.johnson_rows_i32(w, src)
        full = orc.johnson_i32(w)
        if rows is None or full is None or not np.array_equal(rows, full[src]):
            bad.append(f"johnson rows seed {seed}: differ from the full matrix")
        elif not np.array_equal(rows, orc.fw_i32(w)[src]):
            bad.append(f"johnson rows seed {seed}: differ from Floyd-Warshall")
    w = graphgen.er_potential_i32(40, 0.2, 0, 50, 40, seed=9)
    w[3, 7], w[7, 3] = -60, 10
    if orc.johnson_rows_i32(w, [0, 1]) is not None:
        bad.append("johnson rows: negative cycle not reported")
    return bad


ALL_CHECKS = (check_golden, check_brute_force, check_closed_forms, check_invariants, check_fw_vs_dijkstra,
              check_negative_weights, check_dijkstra_csr, check_johnson_rows)


def run_all(orc) -> list[str]:
    bad = []
    for chk in ALL_CHECKS:
        try:
            bad += chk(orc)
        except Exception as e:  # a broken build may also crash a check
            bad.append(f"{chk.__name__} raised {type(e).__name__}: {e}")
    return bad
