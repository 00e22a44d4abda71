"""The C-ABI boundary on a machine without a GPU: the library builds, loads,
exports every symbol the headers declare, and rejects bad arguments before
touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

import min_graph_gb300 as apsp
from min_graph_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libs():
    return mbuild.build()


def declared_functions(header: str):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(apsp_\w+)\s*\(", text)))


@pytest.mark.parametrize("header,lib", [("apsp.h", "libapsp.so"), ("apsp_debug.h", "libapsp.so"),
                                        ("apsp_sparse.h", "libapsp.so"), ("apsp_ooc.h", "libapsp.so"),
                                        ("apsp_peak.h", "libapsp_peak.so")])
def test_every_declared_symbol_is_exported(libs, header, lib):
    names = declared_functions(header)
    assert names, header
    so = ctypes.CDLL(libs[lib])
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, f"{lib} lacks {missing}"


def test_header_constants_match_binding():
    text = open(os.path.join(ROOT, "include", "apsp.h")).read()
    assert re.search(r"#define APSP_INF_I32 0x3FFFFFFF", text)
    assert apsp.INF_I32 == 0x3FFFFFFF
    assert f"#define APSP_TILE {apsp.TILE}" in text
    assert f"#define APSP_MAX_N {apsp.MAX_N}" in text
    assert "APSP_ENEGCYCLE = 6" in text and apsp.ENEGCYCLE == 6
    sparse = open(os.path.join(ROOT, "include", "apsp_sparse.h")).read()
    assert f"#define APSP_SPARSE_MAX_N {apsp.SPARSE_MAX_N}" in sparse


def test_status_strings_and_version(libs):
    lib = apsp.load()
    for code in range(7):
        s = lib.apsp_status_string(code).decode()
        assert s.startswith("APSP_")
    assert lib.apsp_status_string(99).decode() == "unknown apsp status"
    assert apsp.version() == 100


def test_bad_arguments_rejected_without_cuda(libs):
    lib = apsp.load()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    for fn in (lib.apsp_solve, lib.apsp_solve_i32, lib.apsp_solve_f32,
               lib.apsp_solve_host_i32, lib.apsp_solve_host_f32):
        assert fn(None, 5, 5, None) == apsp.EINVAL         # NULL with n > 0
        assert fn(fake, -1, 5, None) == apsp.EINVAL        # n < 0
        assert fn(fake, 6, 5, None) == apsp.EINVAL         # ld < n
        assert fn(fake, apsp.MAX_N + 1, apsp.MAX_N + 1, None) == apsp.EINVAL
        assert fn(None, 0, 0, None) == apsp.OK              # n = 0 is a no-op
    for fn in (lib.apsp_validate_i32, lib.apsp_validate_f32):
        assert fn(fake, 4, 4, None, None) == apsp.EINVAL    # no flags pointer
        assert fn(fake, 4, 3, None, fake) == apsp.EINVAL
    arr = (ctypes.c_void_p * 2)(fake, fake)
    nul = (ctypes.c_void_p * 2)(fake, None)
    for fn in (lib.apsp_solve_host_batch_i32, lib.apsp_solve_host_batch_f32):
        assert fn(arr, arr, -1, 5, 5, None) == apsp.EINVAL    # count < 0
        assert fn(arr, arr, 2, -1, 5, None) == apsp.EINVAL    # n < 0
        assert fn(arr, arr, 2, 6, 5, None) == apsp.EINVAL     # ld < n
        assert fn(arr, arr, 2, apsp.MAX_N + 1, apsp.MAX_N + 1, None) == apsp.EINVAL
        assert fn(None, arr, 2, 5, 5, None) == apsp.EINVAL    # no input array
        assert fn(arr, None, 2, 5, 5, None) == apsp.EINVAL    # no output array
        assert fn(nul, arr, 2, 5, 5, None) == apsp.EINVAL     # a NULL input
        assert fn(arr, nul, 2, 5, 5, None) == apsp.EINVAL     # a NULL output
        assert fn(None, None, 0, 5, 5, None) == apsp.OK       # count = 0 is a no-op
        assert fn(nul, nul, 2, 0, 0, None) == apsp.OK         # so is n = 0
    assert lib.apsp_phase_timing_enable(0) == apsp.OK
    assert lib.apsp_debug_inject_phase3_timeout(0) == apsp.EINVAL
    assert lib.apsp_debug_inject_phase3_timeout(3 * 10**9) == apsp.EINVAL
    assert lib.apsp_debug_inject_grid_timeout(0) == apsp.EINVAL
    assert lib.apsp_debug_inject_grid_timeout(3 * 10**9) == apsp.EINVAL
    assert lib.apsp_debug_fail_next_allocations(-1) == apsp.EINVAL
    assert lib.apsp_debug_fail_next_allocations(1001) == apsp.EINVAL
    assert lib.apsp_debug_fail_next_allocations(0) == apsp.OK


def test_sparse_bad_arguments_rejected_without_cuda(libs):
    lib = apsp.load()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    big = apsp.SPARSE_MAX_N + 1
    assert lib.apsp_solve_sparse_i32(None, 5, 5, 0, None) == apsp.EINVAL
    assert lib.apsp_solve_sparse_i32(fake, 6, 5, 0, None) == apsp.EINVAL
    assert lib.apsp_solve_sparse_i32(fake, big, big, 0, None) == apsp.EINVAL
    assert lib.apsp_solve_sparse_i32(None, 0, 0, 0, None) == apsp.OK
    assert lib.apsp_johnson_csr_i32(None, fake, fake, 5, 0, fake, 5, None) == apsp.EINVAL
    assert lib.apsp_johnson_csr_i32(fake, fake, fake, 5, 0, None, 5, None) == apsp.EINVAL
    assert lib.apsp_johnson_csr_i32(fake, fake, fake, 5, 0, fake, 4, None) == apsp.EINVAL
    assert lib.apsp_johnson_csr_i32(None, None, None, 0, 0, None, 0, None) == apsp.OK
    assert lib.apsp_sssp_delta_i32(fake, fake, fake, 5, fake, 2, 0, fake, 4, None) == apsp.EINVAL
    assert lib.apsp_sssp_delta_i32(fake, fake, fake, 5, None, 2, 0, fake, 5, None) == apsp.EINVAL
    assert lib.apsp_sssp_delta_i32(fake, fake, fake, 5, fake, -1, 0, fake, 5, None) == apsp.EINVAL
    assert lib.apsp_sssp_delta_i32(fake, fake, fake, 5, fake, 0, 0, fake, 5, None) == apsp.OK
    m = ctypes.c_longlong(0)
    assert lib.apsp_csr_count_i32(fake, 4, 4, None, ctypes.byref(m), None) == apsp.EINVAL
    assert lib.apsp_csr_count_i32(fake, 4, 3, fake, ctypes.byref(m), None) == apsp.EINVAL
    assert lib.apsp_csr_fill_i32(fake, 4, 4, fake, None, fake, None) == apsp.EINVAL
    assert lib.apsp_csr_fill_i32(None, 0, 0, None, None, None, None) == apsp.OK
    assert lib.apsp_sssp_i32(None, None, None, 0, 0, 0, None, None) == apsp.OK
    assert lib.apsp_sssp_i32(fake, fake, fake, 5, 5, 0, fake, None) == apsp.EINVAL    # source >= n
    assert lib.apsp_sssp_i32(fake, fake, fake, 5, -1, 0, fake, None) == apsp.EINVAL   # source < 0
    assert lib.apsp_sssp_i32(fake, fake, fake, 5, 0, 0, None, None) == apsp.EINVAL    # no output
    assert lib.apsp_sssp_i32(fake, fake, fake, 5, 0, 0, ctypes.c_void_p(0x1004), None) == apsp.EINVAL  # misaligned
    h = ctypes.c_void_p(0x1234)
    assert lib.apsp_sssp_graph_create(fake, fake, fake, 5, 0, None, None) == apsp.EINVAL   # no handle slot
    assert lib.apsp_sssp_graph_create(None, fake, fake, 5, 0, None, ctypes.byref(h)) == apsp.EINVAL
    assert h.value is None                                                             # cleared on failure
    assert lib.apsp_sssp_graph_create(fake, fake, fake, 0, 0, None, ctypes.byref(h)) == apsp.EINVAL
    assert lib.apsp_sssp_graph_search(None, 0, fake, None) == apsp.EINVAL
    assert lib.apsp_sssp_graph_info(None, None, None, None) == apsp.EINVAL
    assert lib.apsp_sssp_graph_destroy(None) == apsp.OK


def test_python_binding_rejects_non_cuda():
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        apsp.solve(torch.zeros(4, 4, dtype=torch.int32))
    with pytest.raises(ValueError):
        apsp.solve(torch.zeros(4, 5, dtype=torch.int32))


def test_sparse_and_ooc_bindings_check_their_arguments(libs):
    # argument errors raise before any CUDA call
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        apsp.solve_sparse(torch.zeros(4, 4, dtype=torch.int32))            # not on the device
    i64, i32 = torch.zeros(5, dtype=torch.int64), torch.zeros(3, dtype=torch.int32)
    with pytest.raises(TypeError):
        apsp.johnson_csr(i32, i32, i32)                                    # row_ptr not int64
    with pytest.raises(ValueError):
        apsp.johnson_csr(i64, i32, i32)                                    # host tensors
    with pytest.raises(ValueError):
        apsp.sssp(i64, i32, i32, 0)
    with pytest.raises(ValueError):
        apsp.solve_ooc(np.zeros((4, 5), np.int32))                         # not square
    with pytest.raises(ValueError):
        apsp.solve_ooc(np.zeros((6, 6), np.int32)[:, ::2])                 # not contiguous
    with pytest.raises(TypeError):
        apsp.solve_ooc(np.zeros((4, 4), np.int16))                         # unsupported dtype


def test_host_batch_binding_checks_its_matrices(libs):
    # shapes, leading dimensions and dtypes are checked before any CUDA call
    a4 = np.zeros((4, 4), np.int32)
    with pytest.raises(ValueError):
        apsp.solve_host_batch([a4, np.zeros((5, 5), np.int32)])      # sizes differ
    with pytest.raises(ValueError):
        apsp.solve_host_batch([a4], [np.zeros((4, 4), np.float32)])  # dtypes differ
    with pytest.raises(ValueError):
        apsp.solve_host_batch([a4], [])                             # lengths differ
    with pytest.raises(ValueError):
        apsp.solve_host_batch([np.zeros((4, 5), np.int32)])          # not square
    with pytest.raises(TypeError):
        apsp.solve_host_batch([np.zeros((4, 4), np.int64)])          # unsupported dtype
    assert apsp.solve_host_batch([]) == []


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(apsp, "_lib", None)
    monkeypatch.setattr(apsp, "_LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        apsp.load()


def test_workspace_layout_is_16_byte_aligned():
    # Panels are TB x npad entries with npad a multiple of the tile, so every
    # workspace section starts on a 64 KiB boundary.
    for n in (1, 127, 128, 129, 1000, 32768):
        npad = -(-n // apsp.TILE) * apsp.TILE
        assert (apsp.TILE * npad * 4) % 65536 == 0


def test_ooc_arguments_and_block_choice(libs):
    lib = apsp.load()
    fake = ctypes.c_void_p(0x1000)
    for fn in (lib.apsp_solve_ooc_i32, lib.apsp_solve_ooc_f32):
        assert fn(None, 5, 5, 1 << 30, 0, None) == apsp.EINVAL   # NULL with n > 0
        assert fn(fake, 6, 5, 1 << 30, 0, None) == apsp.EINVAL   # ld < n
        assert fn(fake, 5, 5, 1 << 30, 100, None) == apsp.EINVAL  # K not a multiple of 128
        assert fn(fake, 5, 5, 1 << 30, -128, None) == apsp.EINVAL
        assert fn(None, 0, 0, 0, 0, None) == apsp.OK
    # 5 K^2 + 2 K npad elements of 4 bytes must fit the budget
    def need(n, k):
        npad = -(-n // k) * k
        return 4 * (5 * k * k + 2 * k * npad)
    for n, budget in ((1000, 1 << 20), (32768, 1 << 30), (100000, 8 << 30), (300, 1 << 30)):
        k = apsp.ooc_block(n, budget)
        assert k == 0 or (k % 128 == 0 and need(n, k) <= budget), (n, budget, k)
        if k and k < min(16384, -(-n // 128) * 128):
            assert need(n, k + 128) > budget, (n, budget, k)
    assert apsp.ooc_block(300, 1 << 30) == 384          # the whole matrix is one super-block
    assert apsp.ooc_block(100000, 1000) == 0            # not even K = 128 fits
