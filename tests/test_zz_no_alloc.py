"""apsp_solve_noalloc, the solve for callers that may not allocate device
memory (their GPU memory belongs to another allocator, or an allocation's
device-wide synchronisation is not allowed where they call from).  It runs
the library's kernels on a fixed scratch array compiled into libapsp instead
of an allocated workspace.

Calls go straight through the C-ABI (ctypes).  Each case runs two calls in
a row on different graphs, so a call that depended on leftovers of the
previous one would show.  The output must equal apsp_solve's output bit for
bit (int32), and the CPU oracle's: the whole matrix up to n = 1000, 64
seeded Dijkstra rows at the maximum n.  The second call of each case must
leave the device's free memory unchanged (it allocates nothing).
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import graphgen  # noqa: E402
import min_graph_gb300 as apsp  # noqa: E402
import oracle  # noqa: E402

NOALLOC_MAX_N = 8192  # APSP_NOALLOC_MAX_N in include/apsp.h
CANARY = -777


def _entry():
    f = apsp.load().apsp_solve_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _default_solve(w: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(w).cuda()
    apsp.solve(t)
    apsp.stream_check()
    return t.cpu().numpy()


def _noalloc_solve(w: np.ndarray, ld: int, offset: int, err: "torch.Tensor"):
    """Solve w (n x n) in an n x ld device matrix that starts `offset`
    elements into its allocation.  Returns (result, device free bytes before
    the call, after it)."""
    n = w.shape[0]
    flat = torch.full((n * ld + offset,), CANARY, dtype=torch.int32, device="cuda")
    buf = flat[offset:].view(n, ld)
    buf[:, :n].copy_(torch.from_numpy(w))
    stream = torch.cuda.current_stream()
    stream.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    rc = _entry()(buf.data_ptr(), n, ld, stream.cuda_stream, err.data_ptr())
    assert rc == apsp.OK, apsp.status_string(rc)
    stream.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    host = flat.cpu().numpy()
    assert np.all(host[:offset] == CANARY), "wrote before the matrix"
    mat = host[offset:].reshape(n, ld)
    assert np.all(mat[:, n:] == CANARY), "wrote outside the n x n matrix"
    return mat[:, :n], free_before, free_after


def _check_vs_oracle(w: np.ndarray, got: np.ndarray, call: int):
    n = w.shape[0]
    if n <= 1000:
        want = oracle.fw_i32(w, threads=oracle.default_threads())
        rows = np.arange(n)
    else:
        rows = np.random.default_rng(n + call).choice(n, 64, replace=False).astype(np.int32)
        want = oracle.dijkstra_i32(w, rows)
    mism = np.argwhere(got[rows] != want)
    assert mism.size == 0, (f"call {call}: {len(mism)} entries differ from the oracle, first "
                            f"{tuple(mism[0])}: {got[rows][tuple(mism[0])]} vs {want[tuple(mism[0])]}")


# (100, 100): one tile, phase 1 only.  (129, 132) one element past a 16-byte
# boundary: the cp.async phase 3 (no TMA).  (NOALLOC_MAX_N, ...): the maximum.
@pytest.mark.parametrize("n,ld,offset", [(100, 100, 0), (129, 132, 1), (300, 307, 0), (1000, 1000, 0),
                                         (NOALLOC_MAX_N, NOALLOC_MAX_N, 0)])
def test_noalloc_matches_apsp_solve_on_two_calls_in_a_row(n, ld, offset):
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    graphs = [graphgen.er_i32(n, 0.3, 1, 1000, seed=n + 1),   # dense first,
              graphgen.er_i32(n, 0.002, 1, 1000, seed=n + 2)]  # then sparse (many INF)
    for call, w in enumerate(graphs):
        got, free_before, free_after = _noalloc_solve(w, ld, offset, err)
        assert int(err.item()) == 0, f"call {call}: device error word {int(err.item())}"
        if call == 1:
            assert free_after == free_before, (f"call {call}: device free memory changed by "
                                               f"{free_after - free_before} bytes")
        want = _default_solve(w)
        mism = np.argwhere(got != want)
        assert mism.size == 0, (f"call {call}: {len(mism)} entries differ, first {tuple(mism[0])}: "
                                f"{got[tuple(mism[0])]} vs {want[tuple(mism[0])]}")
        _check_vs_oracle(w, got, call)


def test_noalloc_rejects_n_beyond_its_scratch():
    t = torch.zeros(4, dtype=torch.int32, device="cuda")  # never touched: rejected first
    f = _entry()
    assert f(t.data_ptr(), NOALLOC_MAX_N + 1, NOALLOC_MAX_N + 1, None, None) == apsp.EINVAL
    assert f(t.data_ptr(), 5, 4, None, None) == apsp.EINVAL
    assert f(None, 0, 0, None, None) == apsp.OK
