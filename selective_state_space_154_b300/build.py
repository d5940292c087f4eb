"""Build the CUDA library in-tree: nvcc → selective_state_space_154_b300/_lib/libssm_b300.so.

Run as ``python -m selective_state_space_154_b300.build`` (or through
``__graft_entry__.build()``).  Cross-compiles for sm_103a; no GPU is needed.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libssm_b300.so")
# a separate throughput probe of the arithmetic pipes, loaded only by the benchmark
PROBE_SRC = os.path.join(CSRC, "probe", "pipe_rates.cu")
PROBE_PATH = os.path.join(LIB_DIR, "libssm_probe.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-cudart", "shared",
]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) \
        + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build_probe(force: bool = False) -> str:
    if not force and os.path.exists(PROBE_PATH) and os.path.getmtime(PROBE_PATH) > os.path.getmtime(PROBE_SRC):
        return PROBE_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = PROBE_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([NVCC, "-shared", *NVCC_FLAGS, PROBE_SRC, "-o", tmp,
                           "-Xlinker", "-rpath,/usr/local/cuda/lib64"])
    os.replace(tmp, PROBE_PATH)
    return PROBE_PATH


def build(force: bool = False, verbose: bool = False) -> str:
    build_probe(force)
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    from concurrent.futures import ThreadPoolExecutor

    def compile_one(src):
        obj = os.path.join(LIB_DIR, os.path.basename(src) + ".o")
        cmd = [NVCC, *NVCC_FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.check_call(cmd)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([NVCC, "-shared", *NVCC_FLAGS, *objs, "-o", tmp,
                           "-Xlinker", "-rpath,/usr/local/cuda/lib64"])
    os.replace(tmp, LIB_PATH)
    for o in objs:
        os.remove(o)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
