"""apsp_solve_noalloc, the solve for callers that may not allocate device
memory (their GPU memory belongs to another allocator, or an allocation's
device-wide synchronisation is not allowed where they call from).  It runs
the library's kernels on a fixed scratch array compiled into libapsp instead
of an allocated workspace.

Calls go straight through the C-ABI (ctypes).  Each case runs two calls in
a row on different graphs, so a call that depended on leftovers of the
previous one would show.  The output must equal apsp_solve's output bit for
bit (int32), which is how every int32 parity test here compares.
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

NOALLOC_MAX_N = 8192  # APSP_NOALLOC_MAX_N in include/apsp.h


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


def _noalloc_solve(w: np.ndarray, ld: int, err: "torch.Tensor") -> np.ndarray:
    n = w.shape[0]
    canary = -777
    buf = torch.full((n, ld), canary, dtype=torch.int32, device="cuda")
    buf[:, :n].copy_(torch.from_numpy(w))
    stream = torch.cuda.current_stream()
    rc = _entry()(buf.data_ptr(), n, ld, stream.cuda_stream, err.data_ptr())
    assert rc == apsp.OK, apsp.status_string(rc)
    stream.synchronize()
    host = buf.cpu().numpy()
    assert np.all(host[:, n:] == canary), "wrote outside the n x n matrix"
    return host[:, :n]


@pytest.mark.parametrize("n,ld", [(1000, 1000), (300, 307), (NOALLOC_MAX_N, NOALLOC_MAX_N)])
def test_noalloc_matches_apsp_solve_on_two_calls_in_a_row(n, ld):
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    graphs = [graphgen.er_i32(n, 0.3, 1, 1000, seed=n + 1),   # dense first,
              graphgen.er_i32(n, 0.002, 1, 1000, seed=n + 2)]  # then sparse (many INF)
    for call, w in enumerate(graphs):
        got = _noalloc_solve(w, ld, err)
        assert int(err.item()) == 0, f"call {call}: device error word {int(err.item())}"
        want = _default_solve(w)
        mism = np.argwhere(got != want)
        assert mism.size == 0, (f"call {call}: {len(mism)} entries differ, first {tuple(mism[0])}: "
                                f"{got[tuple(mism[0])]} vs {want[tuple(mism[0])]}")


def test_noalloc_rejects_n_beyond_its_scratch():
    t = torch.zeros(4, dtype=torch.int32, device="cuda")  # never touched: rejected first
    f = _entry()
    assert f(t.data_ptr(), NOALLOC_MAX_N + 1, NOALLOC_MAX_N + 1, None, None) == apsp.EINVAL
    assert f(t.data_ptr(), 5, 4, None, None) == apsp.EINVAL
    assert f(None, 0, 0, None, None) == apsp.OK
