"""Builds libflce.so in-tree with nvcc for sm_103a (GB300).

Each .cu file under csrc/ compiles to an object in parallel; the objects
link into linear_cross_entropy_token_gb300/libflce.so. nvcc cross-compiles,
so this runs on a machine without a GPU too.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libflce.so")
SOURCES = ["flce_api.cu", "flce_umma.cu", "flce_rows.cu", "flce_simt.cu", "flce_static.cu"]
HEADERS = ["ptx.cuh", "flce_internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


GEMM_SOURCES = ("flce_umma.cu", "ptx.cuh", "flce_internal.h")


def _code_only(text: str) -> str:
    """C/C++ source with its comments removed and its whitespace collapsed:
    what the compiler sees, so that editing a comment does not change the
    hash. (A "//" inside a string literal also ends the line's code here;
    the kernel sources hold none that matter.)"""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash(names=GEMM_SOURCES) -> str:
    """Short hash of the code (comments and whitespace aside) of CUDA
    sources, by default those of the tcgen05 GEMM kernels: it identifies the
    kernels a profile of them describes."""
    import hashlib
    h = hashlib.sha256()
    for name in sorted(names):
        if os.path.exists(os.path.join(CSRC, name)):
            with open(os.path.join(CSRC, name), encoding="utf-8") as f:
                h.update(name.encode())
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "flce.h"),
                                                     os.path.abspath(__file__)]
    cc = nvcc()
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append([cc, *ARCH, *FLAGS, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(max(1, len(jobs))) as ex:
        logs = list(ex.map(run, jobs))
    if verbose:
        for lg in logs:
            sys.stderr.write(lg)
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        run([cc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
