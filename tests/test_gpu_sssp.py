"""GPU parity of the grid-wide single-source Delta-stepping search
(apsp_sssp_i32, include/apsp_sparse.h) against the oracle's CSR Dijkstra,
element by element (int32, bit-exact).

Inputs: R-MAT graphs (the Delta-stepping page's workload shape, scale up to
20 with 32 arcs per vertex), ER graphs of ragged sizes, graphs built to
exercise the hub paths (a CTA's list of high-degree vertices, and its
overflow), multigraphs, unreachable vertices and zero weights.
"""
import numpy as np
import pytest

import graphgen
import oracle
from gpu_util import INF, assert_i32_exact

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import min_graph_gb300 as apsp  # noqa: E402


def dev(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


def csr_of(w: np.ndarray):
    n = w.shape[0]
    mask = (w < INF) & ~np.eye(n, dtype=bool)
    rows, cols = np.nonzero(mask)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.add.at(row_ptr, rows + 1, 1)
    return np.cumsum(row_ptr), cols.astype(np.int32), w[rows, cols].astype(np.int32)


def check(row_ptr, col, w, sources, delta=0, what=""):
    g = dev(row_ptr, col, w)
    ref = oracle.dijkstra_csr_i32(row_ptr, col, w, sources)
    for q, s in enumerate(sources):
        got = apsp.sssp(*g, int(s), delta=delta).cpu().numpy()
        assert_i32_exact(got, ref[q], f"{what} source {s} delta {delta}")


@pytest.mark.parametrize("scale", [4, 8, 12, 16])
def test_rmat(scale):
    row_ptr, col, w = graphgen.rmat_csr(scale, whi=1000, seed=scale)
    n = 1 << scale
    src = np.random.default_rng(scale).choice(n, min(n, 4), replace=False)
    check(row_ptr, col, w, src, what=f"rmat{scale}")


@pytest.mark.parametrize("n", [1, 2, 31, 33, 1000, 5003])
def test_er_ragged_sizes(n):
    w = graphgen.er_i32(n, min(1.0, 8.0 / max(n, 1)), 0, 500, seed=n)
    check(*csr_of(w), [0, n - 1, n // 2], what=f"er n={n}")


@pytest.mark.parametrize("delta", [1, 13, 1000, 1 << 29, 0])
def test_every_delta_gives_the_same_distances(delta):
    row_ptr, col, w = graphgen.rmat_csr(13, whi=1000, seed=3)
    check(row_ptr, col, w, [0, 77], delta=delta, what="rmat13")


def test_hubs_on_the_cta_list_and_past_its_capacity():
    # every vertex of this dense graph has ~2000 arcs, and all 4096 of them
    # sit in the first CTA's bitmap words: most go past the list capacity
    w = graphgen.er_i32(4096, 0.5, 1, 10000, seed=11)
    check(*csr_of(w), [0, 4095], what="dense er4096")
    # a few hubs in a sparse graph: the list itself
    rng = np.random.default_rng(2)
    n = 20000
    tail = np.concatenate([rng.integers(0, n, 60000), np.repeat([5, 9000, 17000], 5000)])
    head = rng.integers(0, n, tail.size)
    wt = rng.integers(0, 1000, tail.size).astype(np.int32)
    order = np.argsort(tail, kind="stable")
    row_ptr = np.concatenate([[0], np.cumsum(np.bincount(tail, minlength=n))]).astype(np.int64)
    check(row_ptr, head[order].astype(np.int32), wt[order], [5, 123], what="hubs")


def test_multigraph_zero_weights_and_unreachable():
    rng = np.random.default_rng(9)
    n = 3000
    tail = rng.integers(0, n // 2, 20000)  # vertices >= n/2 have no out-arcs
    head = rng.integers(0, n, 20000)
    wt = rng.integers(0, 3, 20000).astype(np.int32)  # many zero weights, parallel arcs, self-loops
    order = np.argsort(tail, kind="stable")
    row_ptr = np.concatenate([[0], np.cumsum(np.bincount(tail, minlength=n))]).astype(np.int64)
    ref = oracle.dijkstra_csr_i32(row_ptr, head[order].astype(np.int32), wt[order], [0, n - 1])
    assert (ref == INF).any()
    check(row_ptr, head[order].astype(np.int32), wt[order], [0, n - 1], what="multigraph")


def test_no_arcs_and_a_single_vertex():
    for n in (1, 40):
        got = apsp.sssp(*dev(np.zeros(n + 1, np.int64), np.zeros(0, np.int32), np.zeros(0, np.int32)), 0)
        ref = np.full(n, INF, np.int32)
        ref[0] = 0
        assert_i32_exact(got.cpu().numpy(), ref, f"no arcs n={n}")


def test_agrees_with_the_per_cta_search():
    row_ptr, col, w = graphgen.rmat_csr(14, whi=5000, seed=21)
    g = dev(row_ptr, col, w)
    src = np.array([0, 3, 999, 16383], dtype=np.int32)
    rows = apsp.sssp_delta(*g, torch.from_numpy(src).cuda()).cpu().numpy()
    for q, s in enumerate(src):
        assert_i32_exact(apsp.sssp(*g, int(s)).cpu().numpy(), rows[q], f"source {s}")


def test_bad_inputs_rejected():
    row_ptr, col, w = graphgen.rmat_csr(6, whi=10, seed=1)
    g = dev(row_ptr, col, w)
    for bad_src in (-1, 64):
        with pytest.raises(apsp.ApspError) as ei:
            apsp.sssp(*g, bad_src)
        assert ei.value.status == apsp.EINVAL
    wneg = g[2].clone()
    wneg[3] = -1
    with pytest.raises(apsp.ApspError) as ei:
        apsp.sssp(g[0], g[1], wneg, 0)
    assert ei.value.status == apsp.EINVAL
    badcol = g[1].clone()
    badcol[0] = 64
    with pytest.raises(apsp.ApspError) as ei:
        apsp.sssp(g[0], badcol, g[2], 0)
    assert ei.value.status == apsp.EINVAL
    out = torch.empty(65, dtype=torch.int32, device="cuda")[1:]  # 4-byte offset: not 16-byte aligned
    with pytest.raises(apsp.ApspError) as ei:
        apsp.sssp(*g, 0, out=out)
    assert ei.value.status == apsp.EINVAL


def test_rmat_scale20_sampled_sources():
    row_ptr, col, w = graphgen.rmat_csr(20)
    check(row_ptr, col, w, [0, 123457], what="rmat20")


def test_prepared_graph_searches():
    row_ptr, col, w = graphgen.rmat_csr(15, whi=3000, seed=5)
    g = dev(row_ptr, col, w)
    graph = apsp.SsspGraph(*g)
    n, m, delta = graph.info()
    assert n == 1 << 15 and m == int(row_ptr[-1]) and delta > 0
    del g  # the prepared graph keeps its own copy
    torch.cuda.empty_cache()
    src = [0, 7, 32767, 12345]
    ref = oracle.dijkstra_csr_i32(row_ptr, col, w, src)
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    for q, s_ in enumerate(src):
        assert_i32_exact(graph.search(s_, out=out).cpu().numpy(), ref[q], f"prepared source {s_}")
    with pytest.raises(apsp.ApspError) as ei:
        graph.search(n)
    assert ei.value.status == apsp.EINVAL
    graph.close()
    graph.close()  # idempotent
    bad = dev(row_ptr, col, -w)
    with pytest.raises(apsp.ApspError) as ei:
        apsp.SsspGraph(*bad)
    assert ei.value.status == apsp.EINVAL


def test_partition_of_a_hub_larger_than_a_warp_pass():
    # a vertex with 300000 arcs takes the one-CTA-per-vertex partition
    rng = np.random.default_rng(8)
    n = 50000
    tail = np.concatenate([rng.integers(0, n, 100000), np.full(300000, 4)])
    head = rng.integers(0, n, tail.size)
    wt = rng.integers(0, 5000, tail.size).astype(np.int32)
    order = np.argsort(tail, kind="stable")
    row_ptr = np.concatenate([[0], np.cumsum(np.bincount(tail, minlength=n))]).astype(np.int64)
    for delta in (0, 1, 2500):
        check(row_ptr, head[order].astype(np.int32), wt[order], [4, 9], delta=delta, what="mega hub")


def test_grid_barrier_timeout_is_reported_and_the_context_survives():
    row_ptr, col, w = graphgen.rmat_csr(12, whi=1000, seed=2)
    g = dev(row_ptr, col, w)
    apsp.debug_inject_grid_timeout(50_000_000)  # 50 ms
    with pytest.raises(apsp.ApspError) as ei:
        apsp.sssp(*g, 0)
    assert ei.value.status == apsp.ETIMEOUT
    check(row_ptr, col, w, [0, 9], what="after a timeout")
    graph = apsp.SsspGraph(*g)
    apsp.debug_inject_grid_timeout(50_000_000)
    with pytest.raises(apsp.ApspError) as ei:
        graph.search(0)
    assert ei.value.status == apsp.ETIMEOUT
    ref = oracle.dijkstra_csr_i32(row_ptr, col, w, [0])[0]
    assert_i32_exact(graph.search(0).cpu().numpy(), ref, "prepared, after a timeout")
    graph.close()
