"""Pins for the CPU oracle (no GPU needed).

The oracle is trusted only because these pass: hand-worked graphs, brute
force over simple paths, closed forms, breadth-first search, shortest-path
invariants, and agreement of two independent algorithms.  The last test
plants typical mistakes in copies of the oracle's C source and checks that
each one makes at least one pin fail.
"""

import numpy as np
import pytest

import graphgen
import oracle
import pins


def _fail_msg(bad):
    return "\n".join(bad[:20])


def test_golden_fixtures():
    assert len(pins.golden_files()) >= 11
    bad = pins.check_golden(oracle.default())
    assert not bad, _fail_msg(bad)


def test_brute_force_small_graphs():
    bad = pins.check_brute_force(oracle.default())
    assert not bad, _fail_msg(bad)


def test_closed_forms():
    bad = pins.check_closed_forms(oracle.default())
    assert not bad, _fail_msg(bad)


def test_invariants():
    bad = pins.check_invariants(oracle.default())
    assert not bad, _fail_msg(bad)


def test_fw_agrees_with_dijkstra():
    bad = pins.check_fw_vs_dijkstra(oracle.default())
    assert not bad, _fail_msg(bad)


def test_negative_weights():
    bad = pins.check_negative_weights(oracle.default())
    assert not bad, _fail_msg(bad)


def test_parallel_fw_identical_to_serial():
    w = graphgen.er_i32(333, 0.02, 1, 1000, 5)
    orc = oracle.default()
    assert np.array_equal(orc.fw_i32(w, threads=1), orc.fw_i32(w, threads=4))
    wf = graphgen.er_f32(333, 0.02, 6)
    assert np.array_equal(orc.fw_f64(wf, threads=1), orc.fw_f64(wf, threads=4))


def test_fw_steps_compose():
    """Running steps [0,a) then [a,n) equals the full run."""
    w = graphgen.er_i32(200, 0.03, 1, 100, 8)
    orc = oracle.default()
    d = np.minimum(w, oracle.INF_I32).astype(np.int32)
    orc.fw_i32_steps(d, 0, 77)
    orc.fw_i32_steps(d, 77, 200, threads=2)
    assert np.array_equal(d, orc.fw_i32(w))


def test_fw_f64_steps_compose():
    """The fp64 steps [0,a) then [a,n) equal the full fp64 run."""
    w = graphgen.er_f32(150, 0.05, 3)
    orc = oracle.default()
    d = w.astype(np.float64)
    orc.fw_f64_steps(d, 0, 60)
    orc.fw_f64_steps(d, 60, 150, threads=2)
    assert np.array_equal(d, orc.fw_f64(w))


def test_networkx_third_opinion():
    nx = pytest.importorskip("networkx")
    for seed, n, p in ((1, 60, 0.05), (2, 90, 0.1)):
        w = graphgen.er_i32(n, p, 1, 50, seed)
        g = nx.DiGraph()
        g.add_nodes_from(range(n))
        for i, j in zip(*np.nonzero((w < oracle.INF_I32) & ~np.eye(n, dtype=bool))):
            g.add_edge(int(i), int(j), weight=int(w[i, j]))
        ref = nx.floyd_warshall_numpy(g, nodelist=range(n), weight="weight")
        ref = np.where(np.isinf(ref), oracle.INF_I32, ref).astype(np.int64)
        assert np.array_equal(oracle.fw_i32(w).astype(np.int64), ref)


def test_johnson_rows():
    bad = pins.check_johnson_rows(oracle.default())
    assert not bad, _fail_msg(bad)


def test_dijkstra_csr():
    bad = pins.check_dijkstra_csr(oracle.default())
    assert not bad, _fail_msg(bad)


def test_generator_rmat_shape():
    # 2^scale vertices, 32 arcs per vertex, deterministic, weights in range,
    # a heavy-tailed out-degree (R-MAT quadrant probabilities 0.57/0.19/0.19/0.05)
    row_ptr, col, w = graphgen.rmat_csr(12, whi=1000)
    n = 1 << 12
    assert row_ptr.shape == (n + 1,) and row_ptr[0] == 0 and row_ptr[-1] == 32 * n
    assert np.all(np.diff(row_ptr) >= 0) and col.min() >= 0 and col.max() < n
    assert w.min() >= 1 and w.max() <= 1000
    deg = np.diff(row_ptr)
    assert deg.max() > 20 * deg.mean() and np.mean(deg == 0) > 0.1
    r2 = graphgen.rmat_csr(12, whi=1000)
    assert all(np.array_equal(a, b) for a, b in zip((row_ptr, col, w), r2))
    # arcs of a row keep the draw order: the counting sort is stable
    assert np.array_equal(graphgen.rmat_csr(12, whi=1000, threads=1)[1], col)


def test_generator_splitmix64_known_value():
    # First output of SplitMix64 seeded with 0 (published reference value).
    assert graphgen.splitmix64_at(0, 1) == 0xE220A8397B1DCDAF


def test_generator_configs_are_the_five_workloads():
    # the five workloads: graph family, size, arc probability or attachment
    # count, weight range and seed, exactly as stated for the benchmark
    c = graphgen.CONFIGS
    assert c["er256"] == {"kind": "er", "n": 256, "p": 0.1, "wlo": 1, "whi": 100, "seed": 1, "dtype": "int32"}
    assert c["er2048"] == {"kind": "er", "n": 2048, "p": 0.05, "wlo": 1, "whi": 1000, "seed": 2, "dtype": "int32"}
    assert c["er8192"] == {"kind": "er", "n": 8192, "p": 0.5, "wlo": 1, "whi": 10000, "seed": 3, "dtype": "int32"}
    assert c["ba16384"] == {"kind": "ba", "n": 16384, "beta": 8, "wlo": 1, "whi": 1000, "seed": 4, "dtype": "int32"}
    assert c["er32768"] == {"kind": "er", "n": 32768, "p": 0.01, "seed": 5, "dtype": "float32"}


def test_generator_shapes():
    w = graphgen.make("er256")
    assert w.shape == (256, 256) and np.all(np.diag(w) == 0)
    off = w[~np.eye(256, dtype=bool)]
    frac = np.mean(off < oracle.INF_I32)
    assert 0.08 < frac < 0.12
    assert off[off < oracle.INF_I32].min() >= 1 and off[off < oracle.INF_I32].max() <= 100
    b = graphgen.ba_i32(2000, 8, 1, 1000, 4)
    arcs = np.count_nonzero(b < oracle.INF_I32) - 2000
    assert arcs == 2 * 8 * (2000 - 8)
    assert np.array_equal(b < oracle.INF_I32, (b < oracle.INF_I32).T)  # two arcs per edge
    f = graphgen.er_f32(500, 0.01, 5)
    fo = f[~np.eye(500, dtype=bool)]
    fin = fo[np.isfinite(fo)]
    assert fin.min() > 0 and fin.max() <= 1.0
    # ld > n leaves the pad columns alone
    pad = np.full((10, 13), -7, dtype=np.int32)
    graphgen.er_i32(10, 0.5, 1, 9, 3, ld=13, out=pad)
    assert np.all(pad[:, 10:] == -7)
    assert np.array_equal(pad[:, :10], graphgen.er_i32(10, 0.5, 1, 9, 3))


# Planted mistakes: (description, original text, replacement).  Each must be
# caught by at least one pin.  Only in-bounds mistakes are planted, so a broken
# build cannot corrupt the test process.
MUTANTS = [
    ("fw: operand D[k][i] instead of D[i][k]",
     "int64_t dik = rowi[k];", "int64_t dik = rowk[i];"),
    ("fw: last intermediate vertex dropped",
     "for (int64_t k = 0; k < n; ++k) {\n        const int32_t* rowk",
     "for (int64_t k = 0; k < n - 1; ++k) {\n        const int32_t* rowk"),
    ("fw: inputs above INF not read as INF",
     "if (d[i * ld + j] > O_INF) d[i * ld + j] = (int32_t)O_INF;", ""),
    ("fw: k innermost (one pass of min-plus squaring)",
     "    for (int64_t k = 0; k < n; ++k) {\n        const int32_t* rowk = d + k * ld;\n"
     "#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1) if (threads > 1)\n"
     "        for (int64_t i = 0; i < n; ++i) {\n            int32_t* rowi = d + i * ld;\n"
     "            int64_t dik = rowi[k];\n            if (dik >= O_INF) continue; /* no path i ~> k yet */\n"
     "            for (int64_t j = 0; j < n; ++j) {\n",
     "    for (int64_t i = 0; i < n; ++i) {\n        int32_t* rowi = d + i * ld;\n"
     "        for (int64_t j = 0; j < n; ++j) {\n            for (int64_t k = 0; k < n; ++k) {\n"
     "            const int32_t* rowk = d + k * ld;\n"
     "            int64_t dik = rowi[k];\n            if (dik >= O_INF) continue;\n"),
    ("fw_f64: operand D[k][i] instead of D[i][k]",
     "double dik = rowi[k];", "double dik = rowk[i];"),
    ("dijkstra: heap sift-up comparison reversed",
     "if (!o_less(h, &h->a[c], &h->a[p])) break;", "if (o_less(h, &h->a[c], &h->a[p])) break;"),
    ("dijkstra: relaxation forgets the distance so far (int)",
     "int64_t nd = di[u] + g->wi[e];", "int64_t nd = g->wi[e];"),
    ("dijkstra: relaxation forgets the distance so far (float)",
     "double nd = df[u] + g->wf[e];", "double nd = g->wf[e];"),
    ("dijkstra: float weight read transposed",
     "g->wf[e] = (double)wf32[i * ld + j];", "g->wf[e] = (double)wf32[j * ld + i];"),
    ("johnson: back-transform sign flipped",
     "const int64_t d = di[j] + h[j] - h[i];", "const int64_t d = di[j] - h[j] + h[i];"),
    ("johnson: reweighting sign flipped",
     "g.wi[e] += h[u] - h[g.dst[e]];", "g.wi[e] += h[g.dst[e]] - h[u];"),
    ("johnson: negative-cycle check disabled",
     "h[u] + w[u * ld + v] < h[v]) {", "h[u] + w[u * ld + v] < h[v] - 2000000000) {"),
    ("bellman-ford: source distance not zero",
     "out[src] = 0;", "out[src] = 1;"),
    ("dijkstra_csr: last arc of every row skipped",
     "for (int64_t e = row_ptr[u]; e < row_ptr[u + 1]; ++e) {", "for (int64_t e = row_ptr[u]; e < row_ptr[u + 1] - 1; ++e) {"),
    ("bfs: a new vertex gets its parent's hop count (no + 1)",
     "hops[v] = hops[u] + 1;", "hops[v] = hops[u];"),
    ("bfs: arcs read transposed",
     "(int64_t)w[u * ld + v] < O_INF && hops[v] < 0", "(int64_t)w[v * ld + u] < O_INF && hops[v] < 0"),
]


def _build_mutant(tmp_path, idx, old, new):
    src = open(oracle.SOURCE).read()
    assert old in src, f"planted mistake {idx} no longer matches the oracle source"
    src = src.replace(old, new, 1)
    c = tmp_path / f"mutant{idx}.c"
    c.write_text(src)
    so = tmp_path / f"libmutant{idx}.so"
    oracle.compile_source(str(c), str(so))
    return oracle.Oracle(oracle.bind(str(so)))


@pytest.mark.parametrize("idx", range(len(MUTANTS)), ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, idx):
    desc, old, new = MUTANTS[idx]
    orc = _build_mutant(tmp_path, idx, old, new)
    bad = pins.run_all(orc)
    assert bad, f"no pin caught the planted mistake: {desc}"
