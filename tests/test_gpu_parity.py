"""GPU parity: libapsp on the GPU against the CPU oracle, element by element.

int32 results must be bit-exact; fp32 results must be within 1e-5 relative
error of the fp64 oracle, with the same +inf pattern and a zero diagonal.
Small cases span several 128 x 128 tiles and ragged tails; the five standard
workloads are checked at full size (the matrix in full where the oracle can
afford it, otherwise on 64 seeded rows and columns from Dijkstra).
"""
import numpy as np
import pytest

import graphgen
import oracle
import pins
from gpu_util import INF, assert_f32_close, assert_i32_exact, gpu_solve, threads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import min_graph_gb300 as apsp  # noqa: E402

SIZES = [1, 2, 3, 15, 16, 17, 100, 127, 128, 129, 255, 256, 257, 300, 520, 1000]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("p", [0.01, 0.1, 0.6])
def test_random_int32_exact(n, p):
    w = graphgen.er_i32(n, p, 1, 1000, seed=1000 + n)
    got, pad_ok = gpu_solve(w)
    assert pad_ok
    assert_i32_exact(got, oracle.fw_i32(w, threads=threads()), f"n={n} p={p}")


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("p", [0.01, 0.1, 0.6])
def test_random_f32_close(n, p):
    w = graphgen.er_f32(n, p, seed=2000 + n)
    got, pad_ok = gpu_solve(w)
    assert pad_ok
    assert_f32_close(got, oracle.fw_f64(w, threads=threads()), f"n={n} p={p}")


@pytest.mark.parametrize("n,ld,offset", [(300, 307, 0), (300, 312, 0), (257, 260, 1),
                                         (129, 129, 3), (640, 644, 0), (383, 1000, 5)])
def test_leading_dimension_alignment_and_pad_untouched(n, ld, offset):
    """ld > n, ld not a multiple of 4, and a base not 16-byte aligned all give
    the same result; nothing outside the n x n window is written."""
    w = graphgen.er_i32(n, 0.05, 1, 500, seed=n + ld)
    got, pad_ok = gpu_solve(w, ld=ld, offset=offset)
    assert pad_ok, "library wrote outside the matrix"
    assert_i32_exact(got, oracle.fw_i32(w, threads=threads()), f"n={n} ld={ld} off={offset}")
    wf = graphgen.er_f32(n, 0.05, seed=n + ld)
    gotf, pad_ok = gpu_solve(wf, ld=ld, offset=offset)
    assert pad_ok
    assert_f32_close(gotf, oracle.fw_f64(wf, threads=threads()), f"f32 n={n} ld={ld}")


def test_entries_above_inf_read_as_inf():
    rng = np.random.default_rng(5)
    w = graphgen.er_i32(400, 0.002, 1, 100, seed=9)  # sparse: many unreachable pairs
    holes = rng.random((400, 400)) < 0.3
    np.fill_diagonal(holes, False)
    big = rng.integers(INF + 1, 2**31 - 1, size=(400, 400), dtype=np.int64).astype(np.int32)
    w2 = np.where(holes & (w == INF), big, w).astype(np.int32)
    got, _ = gpu_solve(w2)
    assert_i32_exact(got, oracle.fw_i32(w, threads=threads()), "clamped inputs")
    assert got.max() == INF


def test_golden_fixtures_on_gpu():
    for path in pins.golden_files():
        if "negative" in pins.golden_flags(path):
            continue  # the blocked FW contract is non-negative weights; the sparse path takes these
        name, dtype, w, d = pins.load_golden(path)
        got, _ = gpu_solve(w)
        if dtype == "int32":
            assert_i32_exact(got, d, name)
        else:
            assert np.array_equal(got.astype(np.float64), d), name


def test_closed_forms_on_gpu():
    rng = np.random.default_rng(77)
    n = 1000  # directed path, 8 tiles with a ragged tail
    wts = rng.integers(0, 1000, size=n - 1)
    w = np.full((n, n), INF, dtype=np.int32)
    np.fill_diagonal(w, 0)
    w[np.arange(n - 1), np.arange(1, n)] = wts
    pref = np.concatenate([[0], np.cumsum(wts)])
    ref = np.where(np.arange(n)[:, None] <= np.arange(n)[None, :], pref[None, :] - pref[:, None], INF)
    got, _ = gpu_solve(w)
    assert_i32_exact(got, ref, "directed path")
    n = 513  # line metric: D = W
    x = rng.integers(0, 10**6, size=n)
    w = np.abs(x[:, None] - x[None, :]).astype(np.int32)
    got, _ = gpu_solve(w)
    assert_i32_exact(got, w, "line metric")


def test_already_closed_matrix_is_a_fixed_point():
    w = graphgen.er_i32(700, 0.02, 1, 100, seed=3)
    once, _ = gpu_solve(w)
    twice, _ = gpu_solve(once)
    assert_i32_exact(twice, once, "idempotent")


# ---------------------------------------------------------------- workloads

def test_workload_er256_full():
    w = graphgen.make("er256")
    got, _ = gpu_solve(w)
    assert_i32_exact(got, oracle.fw_i32(w, threads=threads()), "er256")


def test_workload_er2048_full():
    w = graphgen.make("er2048")
    got, _ = gpu_solve(w)
    ref = oracle.fw_i32(w, threads=threads())
    assert_i32_exact(got, ref, "er2048")


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    s = np.sort(rng.choice(n, size=k, replace=False)).astype(np.int32)
    s[0], s[-1] = 0, n - 1  # always include both ends (first and ragged-last tiles)
    return np.unique(s)


def test_workload_er8192_sampled_rows_and_columns():
    w = graphgen.make("er8192")
    got, _ = gpu_solve(w)
    src = _sample(8192, 64, 8192)
    rows = oracle.dijkstra_i32(w, src, threads=threads())
    cols = oracle.dijkstra_i32(w, src, reverse=True, threads=threads())
    assert_i32_exact(got[src, :], rows, "er8192 rows")
    assert_i32_exact(got[:, src].T, cols, "er8192 columns")
    assert np.all(np.diag(got) == 0)


def test_workload_ba16384_full_matrix():
    """The bench workload: every entry against all-sources Dijkstra."""
    w = graphgen.make("ba16384")
    got, _ = gpu_solve(w)
    ref = oracle.dijkstra_i32(w, np.arange(16384, dtype=np.int32), threads=threads())
    assert_i32_exact(got, ref, "ba16384")


@pytest.mark.parametrize("split", ["1", "4"])
def test_tile_split_over_many_rounds(split, monkeypatch):
    """A forced split on 32 rounds, where the head of ordinary tiles is
    shorter than the ordinary tiles (so every item kind of a launch occurs):
    sampled rows against Dijkstra, and both splits give the same matrix."""
    monkeypatch.setenv("APSP_FUSED_SPLIT", split)
    n = 4000
    w = graphgen.er_i32(n, 0.01, 1, 1000, seed=41)
    got, _ = gpu_solve(w)
    src = np.random.default_rng(41).choice(n, 32, replace=False).astype(np.int32)
    assert_i32_exact(got[src], oracle.dijkstra_i32(w, src), f"split {split} rows")
    monkeypatch.setenv("APSP_FUSED_SPLIT", "2")
    other, _ = gpu_solve(w)
    assert np.array_equal(got, other)


def test_workload_er32768_f32_sampled_rows():
    w = graphgen.make("er32768")
    got, _ = gpu_solve(w)
    src = _sample(32768, 64, 32768)
    ref = oracle.dijkstra_f32(w, src, threads=threads())
    assert_f32_close(got[src, :], ref, "er32768 rows", diag_rows=[(i, int(s)) for i, s in enumerate(src)])
    refc = oracle.dijkstra_f32(w, src[:16], reverse=True, threads=threads())
    assert_f32_close(got[:, src[:16]].T, refc, "er32768 columns",
                     diag_rows=[(i, int(s)) for i, s in enumerate(src[:16])])


def test_maximum_size_n65536_sampled_rows_and_columns():
    """The largest size tested: n = 65536 (a 16 GiB int32 matrix, 512 tiles
    per axis, so the most rounds and the longest flag and counter arrays),
    on 16 seeded rows and 4 columns against Dijkstra."""
    n = 65536
    w = graphgen.er_i32(n, 8.0 / n, 1, 1000, seed=65536, threads=threads())
    d = torch.from_numpy(w).cuda()
    apsp.solve(d)
    apsp.stream_check()
    src = _sample(n, 16, 77)
    idx = torch.from_numpy(src.astype(np.int64)).cuda()
    got_rows = d.index_select(0, idx).cpu().numpy()
    got_cols = d.index_select(1, idx[:4]).cpu().numpy().T
    del d
    torch.cuda.empty_cache()
    assert_i32_exact(got_rows, oracle.dijkstra_i32(w, src, threads=threads()), "n=65536 rows")
    assert_i32_exact(got_cols, oracle.dijkstra_i32(w, src[:4], reverse=True, threads=threads()),
                     "n=65536 columns")


# ---------------------------------------------------------------- API

def test_host_entry_point_matches_device():
    for n, ld in ((1000, 1000), (601, 603)):
        w = graphgen.er_i32(n, 0.03, 1, 100, seed=n)
        buf = np.full((n, ld), -3, dtype=np.int32)
        buf[:, :n] = w
        apsp.solve_host(buf, n=n, ld=ld)
        assert_i32_exact(buf[:, :n], oracle.fw_i32(w, threads=threads()), f"host n={n}")
        assert np.all(buf[:, n:] == -3)
        wf = graphgen.er_f32(n, 0.03, seed=n)
        pinned = torch.from_numpy(wf.copy()).pin_memory()
        apsp.solve_host(pinned)
        assert_f32_close(pinned.numpy(), oracle.fw_f64(wf, threads=threads()), f"host f32 n={n}")


def test_host_batch_matches_oracle():
    # four different problems, one of them twice (inputs may repeat when the
    # outputs differ), a ragged leading dimension with canaries, int32 and fp32
    n, ld = 777, 781
    ws = [graphgen.er_i32(n, p, 1, 100, seed=s) for s, p in ((11, 0.01), (12, 0.05), (13, 0.3))]
    ins = []
    for w in ws + [ws[0]]:
        buf = torch.full((n, ld), -3, dtype=torch.int32).pin_memory()
        buf[:, :n] = torch.from_numpy(w)
        ins.append(buf)
    outs = [torch.full((n, ld), -5, dtype=torch.int32).pin_memory() for _ in ins]
    outs[1] = ins[1]  # one result in place
    apsp.solve_host_batch([x[:, :n] for x in ins], [x[:, :n] for x in outs])  # views: ld > n
    refs = [oracle.fw_i32(w, threads=threads()) for w in ws]
    for b, ref in enumerate(refs + [refs[0]]):
        assert_i32_exact(outs[b][:, :n].numpy(), ref, f"batch problem {b}")
    assert np.all(ins[0][:, :n].numpy() == ws[0])  # inputs only read
    for b in (0, 2, 3):
        assert np.all(outs[b][:, n:].numpy() == -5)
    assert np.all(ins[1][:, n:].numpy() == -3)
    # fp32, in place, odd count, unpinned numpy arrays
    wf = [graphgen.er_f32(300, 0.05, seed=s) for s in (21, 22, 23)]
    bufs = [w.copy() for w in wf]
    apsp.solve_host_batch(bufs)
    for b, w in enumerate(wf):
        assert_f32_close(bufs[b], oracle.fw_f64(w, threads=threads()), f"batch f32 problem {b}")
    # one problem, and none
    one = [graphgen.er_i32(129, 0.1, 1, 50, seed=31)]
    ref = oracle.fw_i32(one[0], threads=threads())
    apsp.solve_host_batch(one)
    assert_i32_exact(one[0], ref, "batch of one")
    assert apsp.solve_host_batch([]) == []


def test_failed_allocation_reports_enomem_and_recovers():
    # A host-side hook fails the next device allocation as a full device
    # would: the solve reports APSP_ENOMEM, leaves the matrix alone, and the
    # next solve allocates and is exact.  A small solve (n <= 512, one
    # cluster) needs no workspace: it succeeds with the hook armed.
    lib = apsp.load()
    w = graphgen.er_i32(600, 0.05, 1, 100, seed=3)
    ref = oracle.fw_i32(w, threads=threads())
    w2 = graphgen.er_i32(700, 0.02, 1, 100, seed=4)
    ref2 = oracle.fw_i32(w2, threads=threads())
    ws = graphgen.er_i32(300, 0.05, 1, 100, seed=5)
    refs = oracle.fw_i32(ws, threads=threads())
    try:
        apsp.release()  # the next dense solve must allocate its workspace
        t = torch.from_numpy(w).cuda()
        assert lib.apsp_debug_fail_next_allocations(1) == apsp.OK
        small = torch.from_numpy(ws).cuda()
        apsp.solve(small)
        apsp.stream_check()
        assert_i32_exact(small.cpu().numpy(), refs, "small solve with the allocation hook armed")
        with pytest.raises(apsp.ApspError) as ei:
            apsp.solve(t)
        assert ei.value.status == apsp.ENOMEM
        assert lib.apsp_last_cuda_error() == 2  # cudaErrorMemoryAllocation
        assert np.array_equal(t.cpu().numpy(), w)
        apsp.solve(t)
        apsp.stream_check()
        assert_i32_exact(t.cpu().numpy(), ref, "solve after a failed allocation")
        # the host entry point: its staging buffer is the first allocation
        apsp.release()
        buf = w2.copy()
        assert lib.apsp_debug_fail_next_allocations(1) == apsp.OK
        with pytest.raises(apsp.ApspError) as ei:
            apsp.solve_host(buf)
        assert ei.value.status == apsp.ENOMEM
        assert np.array_equal(buf, w2)
        apsp.solve_host(buf)
        assert_i32_exact(buf, ref2, "host solve after a failed allocation")
    finally:
        lib.apsp_debug_fail_next_allocations(0)


def test_validator_flags():
    w = graphgen.er_i32(300, 0.05, 1, 100, seed=1)
    t = torch.from_numpy(w).cuda()
    assert apsp.validate(t) == 0
    t[5, 5] = 3
    assert apsp.validate(t) == 1
    t[7, 9] = -2
    assert apsp.validate(t) == 3
    f = torch.from_numpy(graphgen.er_f32(300, 0.05, seed=2)).cuda()
    assert apsp.validate(f) == 0
    f[1, 2] = float("nan")
    assert apsp.validate(f) == 4


@pytest.mark.parametrize("fused", ["1", "0"])
def test_phase_timing_counts_launches(fused, monkeypatch):
    monkeypatch.setenv("APSP_FUSED", fused)
    w = torch.from_numpy(graphgen.er_i32(1000, 0.02, 1, 100, seed=4)).cuda()
    apsp.phase_timing_read()
    apsp.phase_timing_enable(True)
    try:
        apsp.solve(w)
        ms, cnt = apsp.phase_timing_read()
    finally:
        apsp.phase_timing_enable(False)
    nb = -(-1000 // apsp.TILE)
    if fused == "1":
        assert cnt == [0, 0, nb + 1]  # prologue + one launch per round
        ms = ms[2:]
    else:
        assert cnt == [nb, nb, nb]
    assert all(m > 0 for m in ms)


def test_two_streams_share_the_workspace_safely():
    ws = [graphgen.er_i32(900, 0.02, 1, 100, seed=s) for s in (1, 2)]
    ts = [torch.from_numpy(w).cuda() for w in ws]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for t, s in zip(ts, streams):
        apsp.solve(t, stream=s)
    torch.cuda.synchronize()
    for t, w in zip(ts, ws):
        assert_i32_exact(t.cpu().numpy(), oracle.fw_i32(w, threads=threads()), "two streams")


def test_empty_and_single():
    got, pad_ok = gpu_solve(np.zeros((1, 1), np.int32))
    assert pad_ok and got[0, 0] == 0
    t = torch.zeros((0, 0), dtype=torch.int32, device="cuda")
    apsp.solve(t)


# Environment settings that select each schedule / phase-3 kernel.  The
# defaults send n <= 512 to the one-cluster small-matrix kernel; every other
# variant turns that off (APSP_SMALL=0) so that the round schedules are
# exercised at these sizes too.
PHASE3_VARIANTS = [
    {},                                                          # default (one cluster when n <= 512)
    {"APSP_SMALL": "0"},                                         # round-fused schedule
    {"APSP_SMALL": "0", "APSP_FUSED_SPLIT": "1"},                # ... each phase-3 tile one item
    {"APSP_SMALL": "0", "APSP_FUSED_SPLIT": "2"},                # ... split in two along k
    {"APSP_SMALL": "0", "APSP_FUSED_SPLIT": "4"},                # ... split in four along k
    {"APSP_SMALL": "0", "APSP_FUSED_OVERLAP": "0"},              # ... each launch after the previous ends
    {"APSP_SMALL": "0", "APSP_FUSED": "0", "APSP_P3_COLS": "8"},   # three kernels, persistent phase 3
    {"APSP_SMALL": "0", "APSP_FUSED": "0", "APSP_P3_COLS": "4"},   # ... with 512 consumer threads
    {"APSP_SMALL": "0", "APSP_FUSED": "0", "APSP_P3_STAGES": "5"},  # ... with a 5-stage slab ring
    {"APSP_SMALL": "0", "APSP_FUSED": "0", "APSP_PHASE3": "cpasync"},  # ... with the cp.async phase 3
]


@pytest.mark.parametrize("n", [129, 255, 256, 300, 1000, 2100])
def test_all_schedules_and_phase3_kernels_agree(n, monkeypatch):
    """Every schedule and phase-3 kernel gives the oracle's result: the
    one-cluster kernel (n <= 512), the round-fused schedule with each split
    of its phase-3 tiles along k, and the three-kernel schedule with each
    phase-3 kernel."""
    w = graphgen.er_i32(n, 0.02, 1, 1000, seed=n + 7)
    ref = oracle.fw_i32(w, threads=threads())
    wf = graphgen.er_f32(n, 0.02, seed=n + 8)
    reff = oracle.fw_f64(wf, threads=threads())
    unsplit_f = None
    for env in PHASE3_VARIANTS:
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        got, _ = gpu_solve(w)
        gotf, _ = gpu_solve(wf)
        for k in env:
            monkeypatch.delenv(k)
        assert_i32_exact(got, ref, f"{env}")
        assert_f32_close(gotf, reff, f"{env} f32")
        # Without the k-split of phase-2 tiles (whose parts may read values
        # that other parts lowered, and so may round differently), every
        # schedule forms each candidate sum with the same IEEE add, and a
        # minimum is exact in any order: the fused schedule's packed fp32
        # core and the three-kernel schedule's add-then-min core agree bit
        # for bit.  (The one-cluster kernel blocks by 32, not 128, so its
        # sums may associate differently: it is held to the tolerance only.)
        if env.get("APSP_FUSED_SPLIT") == "1" or env.get("APSP_FUSED") == "0":
            if unsplit_f is None:
                unsplit_f = gotf
            else:
                assert np.array_equal(gotf.view(np.int32), unsplit_f.view(np.int32)), f"{env} f32 bits"


@pytest.mark.parametrize("fused", ["1", "0"])
@pytest.mark.parametrize("split", ["1", "4"])
def test_bounded_wait_timeout_each_schedule(fused, split, monkeypatch):
    """The timeout hook works in both schedules (and both tile splits)."""
    monkeypatch.setenv("APSP_FUSED", fused)
    monkeypatch.setenv("APSP_FUSED_SPLIT", split)
    w = graphgen.er_i32(600, 0.02, 1, 100, seed=13)
    t = torch.from_numpy(w).cuda()
    apsp.stream_check()
    apsp.debug_inject_phase3_timeout(50_000_000)
    apsp.solve(t)
    with pytest.raises(apsp.ApspError) as ei:
        apsp.stream_check()
    assert ei.value.status == apsp.ETIMEOUT
    got, _ = gpu_solve(w)
    assert_i32_exact(got, oracle.fw_i32(w, threads=threads()), f"after timeout, fused={fused}")


def test_bounded_wait_timeout_is_reported_and_context_survives():
    """A device-side wait that never completes (the test hook withholds one
    k-slab) ends after its bound; the host sees APSP_ETIMEOUT and the GPU
    context stays usable."""
    w = graphgen.er_i32(600, 0.02, 1, 100, seed=12)
    t = torch.from_numpy(w).cuda()
    apsp.stream_check()
    apsp.debug_inject_phase3_timeout(50_000_000)  # 50 ms
    apsp.solve(t)
    with pytest.raises(apsp.ApspError) as ei:
        apsp.stream_check()
    assert ei.value.status == apsp.ETIMEOUT
    apsp.stream_check()  # the error word was cleared
    got, _ = gpu_solve(w)  # and the next solve is correct
    assert_i32_exact(got, oracle.fw_i32(w, threads=threads()), "after timeout")


SMALL_SIZES = [31, 32, 33, 63, 64, 65, 96, 160, 223, 384, 479, 480, 500, 511, 512, 513]


@pytest.mark.parametrize("n", SMALL_SIZES)
def test_small_cluster_path_around_block_edges(n, monkeypatch):
    """The one-cluster kernel (n <= 512) around its 32-wide block edges, up
    to its limit and one past it (n = 513 goes to the round schedule), with
    dense and sparse graphs, int32 bit-exact and fp32 within tolerance.  The
    round-fused schedule on the same inputs (APSP_SMALL=0) must agree."""
    for p in (0.02, 0.5):
        w = graphgen.er_i32(n, p, 1, 1000, seed=3000 + n)
        ref = oracle.fw_i32(w, threads=threads())
        got, pad_ok = gpu_solve(w, ld=n + 3)
        assert pad_ok
        assert_i32_exact(got, ref, f"small path n={n} p={p}")
        monkeypatch.setenv("APSP_SMALL", "0")
        got_rounds, _ = gpu_solve(w)
        monkeypatch.delenv("APSP_SMALL")
        assert_i32_exact(got_rounds, ref, f"round schedule n={n} p={p}")
        wf = graphgen.er_f32(n, p, seed=4000 + n)
        gotf, pad_ok = gpu_solve(wf, offset=1)
        assert pad_ok
        assert_f32_close(gotf, oracle.fw_f64(wf, threads=threads()), f"small path f32 n={n} p={p}")


def test_small_cluster_path_in_a_captured_graph():
    """The one-cluster launch records into a CUDA graph like the other
    schedules and replays correctly."""
    w = graphgen.er_i32(300, 0.05, 1, 1000, seed=77)
    ref = oracle.fw_i32(w, threads=threads())
    src = torch.from_numpy(w).cuda()
    t = src.clone()
    s = torch.cuda.Stream()
    apsp.solve(t, stream=s)  # first solve outside the capture (one-time set-up)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        apsp.solve(t, stream=s)
    for _ in range(2):
        t.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert_i32_exact(t.cpu().numpy(), ref, "graph replay")
