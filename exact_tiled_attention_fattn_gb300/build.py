"""Build libfattn.so (in-tree) from csrc/*.cu for sm_103a with nvcc.

Usage: ``python -m exact_tiled_attention_fattn_gb300.build [--force]``.
Translation units compile in parallel into ``_build/``; the shared library is
linked next to this file, where ``fattn.py`` loads it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfattn")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return _sources() + hdrs + [os.path.join(INCLUDE, "fattn.h"), os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


# The tensor-core prefill splits its launch registers between warpgroups with
# setmaxnreg, assuming ptxas launches it at this many registers per thread; a
# different count would make the split wait forever, so the build refuses it.
PREFILL_TC_LAUNCH_REGS = 168


def _check_launch_registers(ptxas_log: str):
    counts = []
    lines = ptxas_log.splitlines()
    for i, line in enumerate(lines):
        if "Compiling entry function" in line and "prefill_tc_kernel" in line:
            for nxt in lines[i + 1:i + 4]:
                m = re.search(r"Used (\d+) registers", nxt)
                if m:
                    counts.append(int(m.group(1)))
                    break
    if not counts or any(c != PREFILL_TC_LAUNCH_REGS for c in counts):
        raise RuntimeError(f"prefill_tc_kernel launch registers {counts} != {PREFILL_TC_LAUNCH_REGS}: "
                           "the setmaxnreg split in prefill_tc.cu must be recomputed")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libfattn.so unless it is newer than every source."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *CFLAGS, *ARCH, "-Xptxas=-v", "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        if os.path.basename(src) == "prefill_tc.cu":
            _check_launch_registers(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
