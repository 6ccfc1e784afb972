"""Build libfa.so (the C-ABI attention library) for sm_103a, in tree, and
its debug twin libfa_debug.so (-DFA_DEBUG: device-side bounds checks that
record a failure in the status word and skip the access).

    python -m online_softmax_sm_gb300.build [--force] [--debug]

Each csrc/*.cu is compiled to an object in parallel (nvcc, one -gencode for
compute_103a/sm_103a, -lineinfo), then linked into
online_softmax_sm_gb300/libfa.so.  ptxas resource usage (-Xptxas -v) of each
translation unit goes to _build/<name>.ptxas.txt.  Nothing is rebuilt when
the library is newer than every source and header.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
LIB_DEBUG = os.path.join(PKG, "libfa_debug.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(nvcc: str, src: str, debug: bool = False) -> str:
    name = os.path.splitext(os.path.basename(src))[0]
    out = BUILD_DEBUG if debug else BUILD
    obj = os.path.join(out, name + ".o")
    cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", *(["-DFA_DEBUG"] if debug else []), "-I", INCLUDE, "-I", CSRC,
           "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(out, name + ".ptxas.txt"), "w") as f:
        f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, jobs: int | None = None, debug: bool = False) -> str:
    """Compile and link libfa.so (libfa_debug.so with debug=True); returns its path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and up_to_date(lib):
        return lib
    os.makedirs(BUILD_DEBUG if debug else BUILD, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, debug), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list[str]:
    """Both libraries, the two builds side by side (each compiles its units in parallel)."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        futs = [ex.submit(build, force, None, dbg) for dbg in (False, True)]
        return [f.result() for f in futs]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, debug="--debug" in sys.argv))
