"""Builds libidx.so, the indexer's CUDA library, in place (sm_103a only).

Each translation unit is compiled by its own nvcc process, in parallel, then linked into one
shared library with the CUDA runtime linked statically (the driver is resolved at run time).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

HERE = Path(__file__).resolve().parent
CSRC = HERE / "csrc"
LIB = HERE / "libidx.so"
BUILD = HERE.parent / "_build"
SOURCES = ["logits.cu", "logits_d64.cu", "logits_d192.cu", "logits_h16.cu", "logits_h8.cu",
           "logits_mxfp4.cu", "select.cu", "schedule.cu", "mxfp4.cu", "abi.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, extra: list[str]) -> Path:
    obj = BUILD / (Path(src).stem + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", str(CSRC / src), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose_ptxas: bool = False, extra: list[str] | None = None) -> Path:
    """Compile every .cu for sm_103a and link ``libidx.so`` next to this file."""
    BUILD.mkdir(exist_ok=True)
    extra = list(extra or [])
    if verbose_ptxas:
        extra += ["-Xptxas", "-v"]
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB.with_suffix(".so.tmp")
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *map(str, objs), "-o", str(tmp)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv), file=sys.stderr)
