"""GPU parity of the out-of-core solver (include/apsp_ooc.h): the matrix stays
in host memory and streams through the GPU in K x K super-blocks.  int32
results must be bit-exact to the oracle (and to the in-core solve); fp32
within the 1e-5 relative tolerance of the blocked FW.  Small super-blocks
force many super-rounds and ragged edges."""
import numpy as np
import pytest

import graphgen
import oracle
from gpu_util import INF, assert_f32_close, assert_i32_exact, threads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import min_graph_gb300 as apsp  # noqa: E402


@pytest.mark.parametrize("n,block", [(1000, 128), (777, 256), (1500, 512), (3000, 1024), (129, 128), (1, 128)])
def test_int32_against_oracle(n, block):
    w = graphgen.er_i32(n, min(1.0, 10.0 / n), 1, 1000, seed=500 + n)
    ref = oracle.fw_i32(w, threads=threads())
    got = w.copy()
    apsp.solve_ooc(got, device_bytes=1 << 34, block=block)
    assert_i32_exact(got, ref, f"n={n} K={block}")


def test_pinned_tensor_with_leading_dimension():
    n, ld = 700, 733
    w = graphgen.er_i32(n, 0.02, 0, 500, seed=3, ld=ld)
    w[:, n:] = -4242  # canaries beyond column n
    buf = torch.from_numpy(w).pin_memory()
    view = buf[:, :n]
    apsp.solve_ooc(view, block=256)
    got = buf.numpy()
    assert np.all(got[:, n:] == -4242)
    assert_i32_exact(got[:, :n], oracle.fw_i32(np.ascontiguousarray(w[:, :n]), threads=threads()), "pinned ld")


def test_fp32_within_tolerance():
    n = 1100
    w = graphgen.er_f32(n, 0.01, seed=8)
    got = w.copy()
    apsp.solve_ooc(got, block=256)
    assert_f32_close(got, oracle.fw_f64(w, threads=threads()), "fp32 ooc")


def test_entries_above_inf_are_clamped():
    n = 600
    w = graphgen.er_i32(n, 0.01, 1, 100, seed=4)
    rng = np.random.default_rng(1)
    holes = (w == INF) & (rng.random((n, n)) < 0.5)
    w2 = np.where(holes, rng.integers(INF + 1, 2**31 - 1, size=(n, n), dtype=np.int64), w).astype(np.int32)
    apsp.solve_ooc(w2, block=128)
    assert_i32_exact(w2, oracle.fw_i32(w, threads=threads()), "clamped")


def test_budget_picks_the_block_and_one_block_is_in_core():
    n = 2000
    w = graphgen.er_i32(n, 0.005, 1, 50, seed=12)
    ref = oracle.fw_i32(w, threads=threads())
    budget = 4 * (5 * 384 * 384 + 2 * 384 * 2304)  # exactly K = 384 (npad 2304)
    assert apsp.ooc_block(n, budget) == 384
    got = w.copy()
    apsp.solve_ooc(got, device_bytes=budget)
    assert_i32_exact(got, ref, "K from budget")
    got = w.copy()
    apsp.solve_ooc(got, device_bytes=1 << 34)  # K >= n: a single super-block
    assert_i32_exact(got, ref, "single block")
    with pytest.raises(apsp.ApspError) as ei:
        apsp.solve_ooc(w.copy(), device_bytes=1000)
    assert ei.value.status == apsp.EINVAL


def test_ba16384_equals_the_in_core_solve():
    w = graphgen.make("ba16384")
    d = torch.from_numpy(w).cuda()
    apsp.solve(d)
    apsp.stream_check()
    host = torch.from_numpy(w.copy()).pin_memory()
    apsp.solve_ooc(host, block=4096)
    assert torch.equal(host, d.cpu())
    src = np.array([0, 8191, 16383], dtype=np.int32)
    assert_i32_exact(host.numpy()[src], oracle.dijkstra_i32(w, src), "ba16384 rows")
