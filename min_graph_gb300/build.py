"""Build libapsp.so (and the add-min peak probe library) for sm_103a with nvcc.

Translation units compile in parallel; the result lands in
min_graph_gb300/_build/ (git-ignored).  Run as `python -m min_graph_gb300.build`
or call build().  Nothing here needs a GPU: nvcc cross-compiles.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]

LIBS = {
    "libapsp.so": ["apsp_api.cu", "fw_i32.cu", "fw_f32.cu", "noalloc.cu", "sparse.cu", "ooc.cu"],
    "libapsp_peak.so": ["peak.cu"],
}
HEADERS = ["fw_kernels.cuh", "fw_fused.cuh", "fw_cluster.cuh", "fw_launch.h", "fw_launch_impl.cuh", "mm_core.cuh", "tma.cuh"]


def _newest_input(srcs):
    paths = [os.path.join(CSRC, s) for s in srcs] + [os.path.join(CSRC, h) for h in HEADERS]
    paths += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths if os.path.exists(p))


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if p.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + p.stdout)
    return p.stdout


def lib_path(name: str = "libapsp.so") -> str:
    return os.path.join(OUT, name)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> dict:
    """Compile every library; returns {name: path}.  Rebuilds only when a
    source, header or this script is newer than the library."""
    os.makedirs(OUT, exist_ok=True)
    todo = []
    for name, srcs in LIBS.items():
        if not all(os.path.exists(os.path.join(CSRC, s)) for s in srcs):
            continue
        so = lib_path(name)
        if force or not os.path.exists(so) or os.path.getmtime(so) < _newest_input(srcs):
            todo.append((name, srcs))
    objs = {}

    def compile_one(src):
        obj = os.path.join(OUT, src.replace(".cu", ".o"))
        cmd = [NVCC] + CFLAGS + (["-Xptxas", "-v"] if ptxas_info else []) + \
              ["-c", os.path.join(CSRC, src), "-o", obj]
        out = _run(cmd)
        if verbose or ptxas_info:
            sys.stdout.write(out)
        return src, obj

    srcs = sorted({s for _, ss in todo for s in ss})
    if srcs:
        with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
            for src, obj in ex.map(compile_one, srcs):
                objs[src] = obj
    for name, ss in todo:
        tmp = lib_path(name) + f".tmp{os.getpid()}"
        _run([NVCC] + ARCH + ["-shared", "-o", tmp] + [objs[s] for s in ss] + ["-lpthread", "-ldl", "-lrt"])
        os.replace(tmp, lib_path(name))
    return {name: lib_path(name) for name in LIBS if os.path.exists(lib_path(name))}


if __name__ == "__main__":
    res = build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_info="--ptxas-info" in sys.argv)
    for k, v in res.items():
        print(k, v)
