"""Build libsdm.so in-tree with nvcc for sm_103a (B300).

    python -m sparse_memory_linear_key_b300.build [--verbose-ptxas]
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "lib")
LIB = os.path.join(OUT_DIR, "libsdm.so")
SOURCES = ["sdm_api.cu", "bank_init.cu", "project.cu", "proj_tc.cu", "address.cu", "score_tc.cu",
           "scan_codes.cu", "scan.cu", "scan_step.cu", "scan_static.cu", "slot_stats.cu",
           "gdn_dense.cu", "scan_bwd.cu", "addr_bwd.cu"]
HEADERS = ["sdm_common.cuh", "sdm_internal.h", "scan_math.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    inc = os.path.join(os.path.dirname(HERE), "include", "sdm.h")
    return [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [inc, __file__]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
           "-o", tmp] + [os.path.join(CSRC, s) for s in SOURCES] + ["-lcublas"]
    if ptxas_verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.check_call(cmd, cwd=CSRC)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, ptxas_verbose="--verbose-ptxas" in sys.argv))
