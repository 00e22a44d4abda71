"""Helpers shared by the GPU tests: move matrices to the device, compare
with the oracle."""
from __future__ import annotations

import os

import numpy as np

INF = 0x3FFFFFFF
F32_RTOL = 1e-5   # fp32 tolerance: relative error per entry vs the fp64 oracle


def threads():
    return max(1, os.cpu_count() or 1)


def gpu_solve(w: np.ndarray, ld: int | None = None, offset: int = 0, canary=None):
    """Copy w (n x n) into a device buffer with leading dimension ld (and
    `offset` elements before the matrix), solve there, return (result,
    pad_ok).  pad_ok says whether every element outside the n x n window
    still holds the canary."""
    import torch

    import min_graph_gb300 as apsp

    n = w.shape[0]
    ld = n if ld is None else ld
    dt = torch.int32 if w.dtype == np.int32 else torch.float32
    if canary is None:
        canary = -12345 if dt == torch.int32 else -7.5
    total = offset + max(n, 1) * ld + 8
    buf = torch.full((total,), canary, dtype=dt, device="cuda")
    mat = buf[offset:offset + n * ld].view(n, ld)[:, :n] if n > 0 else buf[:0].view(0, 0)
    if n > 0:
        mat.copy_(torch.from_numpy(w))
    apsp.solve(mat)
    apsp.stream_check()
    host = buf.cpu().numpy()
    mask = np.ones(total, dtype=bool)
    for i in range(n):
        mask[offset + i * ld: offset + i * ld + n] = False
    pad_ok = bool(np.all(host[mask] == canary))
    res = np.array(mat.cpu().numpy(), copy=True) if n > 0 else np.zeros((0, 0), w.dtype)
    return res, pad_ok


def assert_i32_exact(got: np.ndarray, ref: np.ndarray, what: str = ""):
    ref = np.asarray(ref).astype(np.int64)
    got = np.asarray(got).astype(np.int64)
    assert got.shape == ref.shape, what
    bad = np.argwhere(got != ref)
    assert bad.size == 0, (f"{what}: {len(bad)} mismatches, first at {tuple(bad[0])}: "
                           f"got {got[tuple(bad[0])]} want {ref[tuple(bad[0])]}")


def assert_f32_close(got: np.ndarray, ref: np.ndarray, what: str = "", diag_rows=None):
    """Relative error <= F32_RTOL where finite, identical +inf pattern, and
    an exactly zero diagonal (diag_rows: row index -> column of the diagonal
    entry, for sampled rows)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, what
    gi, ri = np.isinf(got), np.isinf(ref)
    assert np.array_equal(gi, ri), f"{what}: INF pattern differs at {np.argwhere(gi != ri)[:3]}"
    assert not np.isnan(got).any(), f"{what}: NaN in result"
    fin = ~ri
    err = np.abs(got[fin] - ref[fin])
    tol = F32_RTOL * np.abs(ref[fin])
    if err.size:
        worst = int(np.argmax(err - tol))
        assert np.all(err <= tol), (f"{what}: relative error {err[worst] / max(abs(ref[fin][worst]), 1e-300):.3g}"
                                    f" > {F32_RTOL}")
    if diag_rows is None:
        assert np.all(np.diag(got) == 0.0), f"{what}: non-zero diagonal"
    else:
        for r, c in diag_rows:
            assert got[r, c] == 0.0, f"{what}: non-zero diagonal at source {c}"
