"""Binding of libapsp_peak.so: measured issue rate of the relaxation step
(the compute roofline of the min-plus update).  See include/apsp_peak.h."""
from __future__ import annotations

import ctypes
import os

_SO = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libapsp_peak.so")
_lib = None

VARIANTS = {
    0: "int32 fused add-min (__viaddmin_s32)",
    1: "int32 add then min",
    2: "int32 two relaxations per three-input min (__vimin3_s32)",
    3: "fp32 fminf(acc, a+b)",
    4: "fp32 fminf(acc, fminf(a0+b0, a1+b1))",
    5: "int32 multiply-add adds, three-input integer min",
    6: "int32 adds, fp32 three-input min on bit patterns",
    7: "int32 multiply-add adds, fp32 three-input min on bit patterns",
    8: "core: int32 fused add-min, one k per step (smem-fed)",
    9: "core: int32 two adds + three-input min (smem-fed)",
    10: "core: int32 64-bit packed add + three-input min (smem-fed)",
    11: "core: fp32 add + min, one k per step (smem-fed)",
    12: "core: fp32 two adds + three-input min (smem-fed)",
    13: "core: fp32 add.f32x2 + three-input min (smem-fed)",
    14: "core: int32 fused, compiled for 2 blocks/SM",
    15: "core: fp32 add.f32x2 + min3, compiled for 2 blocks/SM",
    16: "core: int32 mixed, 2/8 rows fused add-min, rest adds + min3",
    17: "core: int32 mixed, 3/8 rows fused add-min, rest adds + min3",
    18: "core: int32 mixed, 2/8 rows fused, rest multiply-add adds + min3",
    19: "core: int32 mixed, 3/8 rows fused, rest multiply-add adds + min3",
    20: "core: int32 mixed, 4/8 rows fused, rest multiply-add adds + min3",
}


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            raise RuntimeError(f"{_SO} not built; run `python -m min_graph_gb300.build`")
        lib = ctypes.CDLL(_SO)
        lib.apsp_peak_addmin.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_longlong)]
        lib.apsp_peak_addmin.restype = ctypes.c_int
        lib.apsp_peak_variants.argtypes = []
        lib.apsp_peak_variants.restype = ctypes.c_int
        lib.apsp_peak_l2_read.argtypes = [ctypes.c_longlong, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        lib.apsp_peak_l2_read.restype = ctypes.c_int
        _lib = lib
    return _lib


def measure(variant: int, blocks: int, threads: int = 256, iters: int = 4096) -> dict:
    """Run one variant; returns relaxations per SM-clock per SM, ms, total."""
    rpc, ms, tot = ctypes.c_double(), ctypes.c_double(), ctypes.c_longlong()
    rc = _load().apsp_peak_addmin(variant, blocks, threads, iters, ctypes.byref(rpc),
                                  ctypes.byref(ms), ctypes.byref(tot))
    if rc != 0:
        raise RuntimeError(f"apsp_peak_addmin({variant}) failed: {rc}")
    return {"variant": variant, "what": VARIANTS[variant], "relax_per_clk_sm": rpc.value,
            "ms": ms.value, "relax": tot.value,
            "relax_per_s": tot.value / (ms.value * 1e-3) if ms.value > 0 else 0.0}


def l2_read(nbytes: int = 64 << 20, blocks: int = 0, threads: int = 256, passes: int = 200) -> dict:
    """L2 read bandwidth (GB/s) over an L2-resident buffer (include/apsp_peak.h).
    blocks = 0 takes 4 per SM of the current device."""
    if blocks <= 0:
        import torch

        blocks = 4 * torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    gbs, ms = ctypes.c_double(), ctypes.c_double()
    rc = _load().apsp_peak_l2_read(int(nbytes), int(blocks), int(threads), int(passes),
                                   ctypes.byref(gbs), ctypes.byref(ms))
    if rc != 0:
        raise RuntimeError(f"apsp_peak_l2_read failed: {rc}")
    return {"bytes": nbytes, "blocks": blocks, "threads": threads, "passes": passes,
            "gbs": gbs.value, "ms": ms.value}
