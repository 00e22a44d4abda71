"""GPU parity of the sparse path (include/apsp_sparse.h): Johnson's APSP with
Delta-stepping searches, the CSR builder and the multi-source search, against
the CPU oracle element by element.  Every result is int32 and must be
bit-exact.

The oracle sides: Floyd-Warshall and Johnson (Bellman-Ford + Dijkstra) for
whole matrices, per-source Dijkstra for sampled rows of the large workloads,
and hand-worked golden fixtures, including negative arc weights and a
negative cycle.
"""
import numpy as np
import pytest

import graphgen
import oracle
import pins
from gpu_util import INF, assert_i32_exact, threads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import min_graph_gb300 as apsp  # noqa: E402


def sparse_solve(w: np.ndarray, delta: int = 0, ld: int | None = None) -> np.ndarray:
    n = w.shape[0]
    ld = n if ld is None else ld
    buf = torch.full((max(n, 1), max(ld, 1)), -777, dtype=torch.int32, device="cuda")
    mat = buf[:n, :n]
    if n:
        mat.copy_(torch.from_numpy(w))
    apsp.solve_sparse(mat, delta=delta)
    host = buf.cpu().numpy()
    if ld > n:
        assert np.all(host[:n, n:] == -777), "columns n..ld-1 were written"
    return np.array(host[:n, :n], copy=True)


def csr_of(w: np.ndarray):
    """CSR of a dense matrix by definition: off-diagonal entries below INF,
    row by row in column order."""
    n = w.shape[0]
    mask = (w < INF) & ~np.eye(n, dtype=bool)
    rows, cols = np.nonzero(mask)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.add.at(row_ptr, rows + 1, 1)
    return np.cumsum(row_ptr), cols.astype(np.int32), w[rows, cols].astype(np.int32)


def dev(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


def to_dev(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


@pytest.mark.parametrize("n", [1, 2, 3, 31, 32, 33, 100, 300, 1000])
@pytest.mark.parametrize("p", [0.005, 0.05, 0.5])
def test_nonnegative_matches_floyd_warshall(n, p):
    w = graphgen.er_i32(n, p, 0, 1000, seed=3000 + n)  # zero weights included
    assert_i32_exact(sparse_solve(w), oracle.fw_i32(w, threads=threads()), f"n={n} p={p}")


@pytest.mark.parametrize("n", [2, 50, 257, 777])
@pytest.mark.parametrize("p", [0.02, 0.3])
def test_negative_weights_match_johnson_oracle(n, p):
    w = graphgen.er_potential_i32(n, p, 0, 1000, 5000, seed=4000 + n)
    assert (w < 0).any() or n == 2
    ref = oracle.johnson_i32(w, threads=threads())
    assert ref is not None
    assert_i32_exact(sparse_solve(w), ref, f"n={n} p={p}")


def test_golden_fixtures():
    for path in pins.golden_files():
        flags = pins.golden_flags(path)
        name, dtype, w, d = pins.load_golden(path)
        if dtype != "int32":
            continue
        if "negative_cycle" in flags:
            t = torch.from_numpy(w).cuda()
            before = t.clone()
            with pytest.raises(apsp.ApspError) as ei:
                apsp.solve_sparse(t)
            assert ei.value.status == apsp.ENEGCYCLE, name
            assert torch.equal(t, before), f"{name}: matrix changed on a negative cycle"
            continue
        assert_i32_exact(sparse_solve(w), d, name)


@pytest.mark.parametrize("delta", [1, 7, 100, 1000, 1 << 29, 0])
def test_every_delta_gives_the_same_distances(delta):
    w = graphgen.er_i32(600, 0.02, 1, 1000, seed=77)
    assert_i32_exact(sparse_solve(w, delta=delta), oracle.fw_i32(w, threads=threads()), f"delta={delta}")


def test_leading_dimension_and_unreached():
    w = graphgen.er_i32(333, 0.003, 1, 50, seed=5)  # many unreachable pairs
    got = sparse_solve(w, ld=400)
    assert_i32_exact(got, oracle.fw_i32(w, threads=threads()), "ld=400")
    assert (got == INF).any()


def test_no_arcs_and_tiny():
    for n in (1, 5, 40):
        w = np.full((n, n), INF, dtype=np.int32)
        np.fill_diagonal(w, 0)
        assert_i32_exact(sparse_solve(w), w, f"empty n={n}")
    t = torch.zeros((0, 0), dtype=torch.int32, device="cuda")
    apsp.solve_sparse(t)


def test_saturation_at_inf_matches_fw():
    # a chain whose prefix sums cross INF: pairs at or beyond INF read INF
    n = 6
    w = np.full((n, n), INF, dtype=np.int32)
    np.fill_diagonal(w, 0)
    for i in range(n - 1):
        w[i, i + 1] = INF // 3 + 1
    ref = oracle.fw_i32(w)
    assert_i32_exact(sparse_solve(w), ref, "saturation")
    assert ref[0, 3] == INF and ref[0, 2] < INF


def test_negative_values_near_the_range_limit():
    # w = w0 + p(i) - p(j) with potentials up to 2^28: the reweighted
    # distances approach 2 * 2^28 and the mapped-back ones go well below 0.
    w = graphgen.er_potential_i32(500, 0.05, 0, 1 << 20, 1 << 28, seed=99)
    ref = oracle.johnson_i32(w, threads=threads())
    assert ref is not None and ref.min() < -(1 << 26)
    assert_i32_exact(sparse_solve(w), ref, "large potentials")


def test_negative_cycle_detected_in_a_large_graph():
    w = graphgen.er_potential_i32(2000, 0.01, 0, 100, 1000, seed=8)
    assert oracle.johnson_i32(w, threads=threads()) is not None
    w2 = w.copy()
    w2[100, 1500], w2[1500, 100] = -10, 5  # a 2-cycle of weight -5
    assert oracle.johnson_i32(w2, threads=threads()) is None
    t = torch.from_numpy(w2).cuda()
    with pytest.raises(apsp.ApspError) as ei:
        apsp.solve_sparse(t)
    assert ei.value.status == apsp.ENEGCYCLE


def test_distances_below_the_range_are_rejected():
    n = 4  # chain 0 -> 1 -> 2 -> 3 of weight -(INF/2) each: d(0,3) < -INF
    w = np.full((n, n), INF, dtype=np.int32)
    np.fill_diagonal(w, 0)
    for i in range(n - 1):
        w[i, i + 1] = -(INF // 2)
    t = torch.from_numpy(w).cuda()
    with pytest.raises(apsp.ApspError) as ei:
        apsp.solve_sparse(t)
    assert ei.value.status == apsp.EINVAL
    w[0, 1] = -INF  # a weight at -INF itself
    with pytest.raises(apsp.ApspError) as ei:
        apsp.solve_sparse(torch.from_numpy(w).cuda())
    assert ei.value.status == apsp.EINVAL


def test_csr_builder_exact():
    for n, p in ((1, 0.5), (37, 0.3), (1000, 0.02), (3000, 0.001)):
        w = graphgen.er_potential_i32(n, p, 0, 100, 50, seed=n)
        rp, col, wt = csr_of(w)
        grp, gcol, gw = apsp.csr_from_dense(torch.from_numpy(w).cuda())
        assert np.array_equal(grp.cpu().numpy(), rp), n
        assert np.array_equal(gcol.cpu().numpy(), col), n
        assert np.array_equal(gw.cpu().numpy(), wt), n


def test_johnson_csr_with_parallel_arcs_and_self_loops():
    rng = np.random.default_rng(4)
    n = 300
    w = graphgen.er_potential_i32(n, 0.03, 0, 500, 300, seed=12)
    rp, col, wt = csr_of(w)
    # add arcs (some parallel to existing ones) and non-negative self-loops,
    # then shuffle each row's order.  Every distance here is >= -300 (the
    # potentials lie in [0, 300]), so extra arcs of weight > 300 close no
    # negative cycle.
    extra_u = rng.integers(0, n, 400)
    extra_v = rng.integers(0, n, 400)
    extra_w = rng.integers(301, 2000, 400).astype(np.int32)
    loops = np.arange(0, n, 7)
    us = np.concatenate([np.repeat(np.arange(n), np.diff(rp)), extra_u, loops])
    vs = np.concatenate([col, extra_v, loops]).astype(np.int32)
    ws = np.concatenate([wt, extra_w, np.full(loops.size, 3, np.int32)]).astype(np.int32)
    order = np.lexsort((rng.random(us.size), us))
    us, vs, ws = us[order], vs[order], ws[order]
    row_ptr = np.concatenate([[0], np.cumsum(np.bincount(us, minlength=n))]).astype(np.int64)
    dense = np.full((n, n), INF, dtype=np.int64)
    np.fill_diagonal(dense, 0)
    off = us != vs
    np.minimum.at(dense, (us[off], vs[off]), ws[off])
    ref = oracle.johnson_i32(dense.astype(np.int32), threads=threads())
    assert ref is not None
    out = torch.full((n, n + 5), -1, dtype=torch.int32, device="cuda")[:, :n]
    got = apsp.johnson_csr(*to_dev(row_ptr, vs, ws), out=out)
    assert_i32_exact(got.cpu().numpy(), ref, "johnson_csr")


def test_negative_self_loop_is_a_negative_cycle():
    row_ptr = np.array([0, 1, 2], dtype=np.int64)
    col = np.array([1, 1], dtype=np.int32)
    wt = np.array([4, -1], dtype=np.int32)  # arc 0->1 and the loop 1->1 of weight -1
    with pytest.raises(apsp.ApspError) as ei:
        apsp.johnson_csr(*to_dev(row_ptr, col, wt))
    assert ei.value.status == apsp.ENEGCYCLE


def test_malformed_csr_rejected():
    col, wt = np.array([1, 0], np.int32), np.array([1, 1], np.int32)
    src = torch.tensor([0], dtype=torch.int32, device="cuda")
    cases = [
        (np.array([0, 1, 1], np.int64), np.array([2], np.int32), np.array([1], np.int32)),  # head >= n
        (np.array([0, 2, 1], np.int64), col, wt),                                            # decreasing
        (np.array([1, 1, 2], np.int64), col, wt),                                            # row_ptr[0] != 0
    ]
    for rp, c, ww in cases:
        for call in (lambda a: apsp.johnson_csr(*a), lambda a: apsp.sssp_delta(*a, src)):
            with pytest.raises(apsp.ApspError) as ei:
                call(to_dev(rp, c, ww))
            assert ei.value.status == apsp.EINVAL, rp


def test_sssp_delta_rows_and_bad_sources():
    w = graphgen.er_i32(1500, 0.01, 0, 300, seed=31)
    rp, col, wt = to_dev(*csr_of(w))
    src = np.array([0, 1499, 7, 7, 800], dtype=np.int32)
    got = apsp.sssp_delta(rp, col, wt, torch.from_numpy(src).cuda())
    assert_i32_exact(got.cpu().numpy(), oracle.dijkstra_i32(w, src), "sssp rows")
    with pytest.raises(apsp.ApspError) as ei:
        apsp.sssp_delta(rp, col, wt, torch.tensor([3, 1500], dtype=torch.int32, device="cuda"))
    assert ei.value.status == apsp.EINVAL
    wneg = wt.clone()
    wneg[0] = -1
    with pytest.raises(apsp.ApspError) as ei:
        apsp.sssp_delta(rp, col, wneg, torch.tensor([0], dtype=torch.int32, device="cuda"))
    assert ei.value.status == apsp.EINVAL


def test_er2048_full_matrix():
    w = graphgen.make("er2048")
    assert_i32_exact(sparse_solve(w), oracle.fw_i32(w, threads=threads()), "er2048")


def test_ba16384_full_matrix_against_dijkstra():
    w = graphgen.make("ba16384")
    got = sparse_solve(w)
    ref = oracle.dijkstra_i32(w, np.arange(w.shape[0], dtype=np.int32))
    assert_i32_exact(got, ref, "ba16384")


def test_ba16384_sparse_equals_blocked_fw():
    w = graphgen.make("ba16384")
    a = torch.from_numpy(w).cuda()
    b = a.clone()
    apsp.solve(a)
    apsp.stream_check()
    apsp.solve_sparse(b)
    assert torch.equal(a, b)


def test_er32768_sampled_sources():
    # the largest n the sparse path takes: int32 weights on the er32768 graph
    # shape (n = 32768, p = 0.01), 64 sampled sources against Dijkstra
    n = apsp.SPARSE_MAX_N
    w = graphgen.er_i32(n, 0.01, 1, 1000, seed=5)
    rp, col, wt = to_dev(*csr_of(w))
    src = np.random.default_rng(1).choice(n, 64, replace=False).astype(np.int32)
    got = apsp.sssp_delta(rp, col, wt, torch.from_numpy(src).cuda())
    assert_i32_exact(got.cpu().numpy(), oracle.dijkstra_i32(w, src), "er32768 rows")


def test_sparse_timing_counts_searches_and_kernels():
    w = graphgen.er_i32(700, 0.02, 1, 100, seed=3)
    t = torch.from_numpy(w).cuda()
    apsp.sparse_timing_read()
    apsp.sparse_timing_enable(True)
    try:
        apsp.solve_sparse(t)
    finally:
        apsp.sparse_timing_enable(False)
    ms, searches, kernels = apsp.sparse_timing_read()
    assert searches == 1 and ms > 0
    assert kernels == 6  # count + scan + fill + weight range + partition + search
    assert apsp.sparse_timing_read() == (0.0, 0, 0)


def test_l2_probe_reports_a_bandwidth():
    import min_graph_gb300.peak as peak

    r = peak.l2_read(8 << 20, passes=4)
    assert r["gbs"] > 100.0


def test_dense_rows_take_the_cta_partition():
    # 9000 vertices with ~8500 arcs each: rows above 8192 arcs are partitioned
    # one CTA per vertex; four searches against Dijkstra rows
    w = graphgen.er_i32(9000, 0.95, 1, 1000, seed=40)
    rp, col, wt = dev(*csr_of(w))
    src = np.array([0, 1, 4500, 8999], dtype=np.int32)
    got = apsp.sssp_delta(rp, col, wt, torch.from_numpy(src).cuda())
    assert_i32_exact(got.cpu().numpy(), oracle.dijkstra_i32(w, src), "dense rows")


@pytest.mark.parametrize("n", [1000, 4000, 8192])
def test_low_degree_graphs_take_narrow_search_ctas(n):
    # at most 8192 vertices, mean degree <= 512 and as many sources as search
    # slots: the 256-thread search kernel (8192 = its largest n); negative
    # weights go through the reweighting; rows against the oracle's Johnson
    w = graphgen.er_potential_i32(n, 8.0 / n, 0, 1000, 2000, seed=n)
    src = np.array([0, 1, n // 2, n - 1], dtype=np.int32)
    ref = oracle.johnson_rows_i32(w, src)
    assert ref is not None and (w[w < INF] < 0).any()
    t = torch.from_numpy(w).cuda()
    apsp.solve_sparse(t)
    got = t[torch.from_numpy(src).long().cuda()].cpu().numpy()
    assert_i32_exact(got, ref, f"n={n} narrow CTAs")


def test_narrow_search_ctas_for_many_sources():
    # 2000 sources of a 3000-vertex graph of mean degree 9, multi-source entry
    w = graphgen.er_i32(3000, 0.003, 0, 300, seed=41)
    rp, col, wt = to_dev(*csr_of(w))
    src = np.random.default_rng(5).integers(0, 3000, 2000).astype(np.int32)
    got = apsp.sssp_delta(rp, col, wt, torch.from_numpy(src).cuda())
    assert_i32_exact(got.cpu().numpy(), oracle.dijkstra_i32(w, src), "2000 sources")


def test_negative_weights_above_the_512_thread_limit():
    # n = 17000 takes the 1024-thread search kernel; rows against the
    # oracle's Johnson for sampled sources
    n = 17000
    w = graphgen.er_potential_i32(n, 0.002, 0, 1000, 2000, seed=77)
    src = np.array([0, 1, 8500, 16999], dtype=np.int32)
    ref = oracle.johnson_rows_i32(w, src)
    assert ref is not None and (w[w < INF] < 0).any()
    t = torch.from_numpy(w).cuda()
    apsp.solve_sparse(t)
    got = t[torch.from_numpy(src).long().cuda()].cpu().numpy()
    assert_i32_exact(got, ref, "n=17000 negative weights")
