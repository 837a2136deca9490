"""Build the CUDA library libexact_attn.so in-tree for sm_103a.

Each .cu translation unit is compiled by nvcc in parallel, then linked into a
shared library under ``exact_attention_tma_gb300/lib/``.  Run as
``python -m exact_attention_tma_gb300.build`` or through
``__graft_entry__.build()``.  Set EA_PTXAS_VERBOSE=1 to print register and
shared-memory usage (``-Xptxas -v``).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(OUT_DIR, "libexact_attn.so")
SOURCES = ["attn_api.cu", "fwd_sm103a.cu", "decode_sm103a.cu", "decode_gqa_mma_sm103a.cu",
           "bwd_sm103a.cu", "fwd_fp8_sm103a.cu", "decode_noalloc.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")
    return cand


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", INCLUDE, "-I", CSRC]
    if os.environ.get("EA_PTXAS_VERBOSE") == "1":
        flags += ["-Xptxas", "-v"]
    tag = f".{os.getpid()}"

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT_DIR, src.replace(".cu", tag + ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or res.returncode != 0 or os.environ.get("EA_PTXAS_VERBOSE") == "1":
            sys.stderr.write(res.stdout + res.stderr)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = os.path.join(OUT_DIR, f"tmp{tag}.so")
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    for o in objs:
        os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
