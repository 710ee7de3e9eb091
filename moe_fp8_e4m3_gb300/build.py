"""Builds the CUDA library ``libfg.so`` in-tree for sm_103a with nvcc.

The translation units compile in parallel; ``-Xptxas -v`` output goes to
``_build/ptxas.log`` and the build fails if any kernel spills registers or uses local
memory."""
from __future__ import annotations

import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfg.so")
SOURCES = ["fg_api.cu", "fg_gemm_nt.cu", "fg_gemm_split.cu", "fg_gemm_tn.cu", "fg_gemm_layouts.cu",
           "fg_gemm_sepc.cu", "fg_gemm_dense.cu", "fg_gemm_swiglu.cu", "fg_gemm_fp4.cu", "fg_gemm_fp4_grouped.cu",
           "fg_mqa.cu", "fg_quant.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags() -> list[str]:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "fg.h"),
                                                                 os.path.abspath(__file__)]
    return any(os.path.getmtime(f) > t for f in deps)


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    cmd = [_nvcc()] + _flags() + ["-Xptxas", "-v", "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
    return obj, r.stderr


def check_ptxas(log: str) -> None:
    bad = []
    for m in re.finditer(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", log):
        if any(int(x) for x in m.groups()):
            bad.append(m.group(0))
    if bad:
        raise RuntimeError("register spills / local memory in kernels: " + "; ".join(bad))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    log = "\n".join(r[1] for r in results)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write(log)
    check_ptxas(log)
    tmp = LIB + ".tmp"
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + [r[0] for r in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    if verbose:
        print(log)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
