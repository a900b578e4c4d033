"""Build the CUDA library ``_lib/libckv.so`` for sm_103a (in-tree, no cmake).

Translation units are compiled in parallel with nvcc / g++ and linked with
``nvcc -shared``.  Only one ``-gencode`` target is emitted: GB300 (sm_103a).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libckv.so")

GENCODE = "-gencode=arch=compute_103a,code=sm_103a"
CUDA_SOURCES = ["kpool.cu", "c128.cu", "prefill_tma.cu", "planner_device.cu", "validate.cu", "probe.cu", "capi.cu"]
CXX_SOURCES = ["planner.cpp"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libckv")


def _sources():
    return [os.path.join(CSRC, s) for s in CUDA_SOURCES + CXX_SOURCES] + [
        os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))
    ] + [os.path.join(INCLUDE, "ckv.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources())


def _compile(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", f"-I{INCLUDE}", f"-I{CSRC}"]
    cmds, objs = [], []
    for s in CUDA_SOURCES:
        o = os.path.join(BUILD, s + ".o")
        cmd = [nvcc, GENCODE, "-lineinfo", *common, "-Xcompiler", "-fPIC", "-c",
               os.path.join(CSRC, s), "-o", o]
        if verbose_ptxas:
            cmd.insert(1, "-Xptxas=-v")
        cmds.append(cmd)
        objs.append(o)
    for s in CXX_SOURCES:
        o = os.path.join(BUILD, s + ".o")
        cmds.append(["g++", "-O2", "-std=c++17", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}",
                     "-I/usr/local/cuda/include", "-c", os.path.join(CSRC, s), "-o", o])
        objs.append(o)
    with cf.ThreadPoolExecutor(max_workers=jobs or len(cmds)) as ex:
        logs = list(ex.map(_compile, cmds))
    if verbose_ptxas:
        sys.stderr.write("".join(logs))
    tmp = LIB + f".tmp{os.getpid()}"
    _compile([nvcc, GENCODE, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
