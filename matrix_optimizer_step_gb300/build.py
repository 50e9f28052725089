"""Build ``libdmuon.so`` in-tree for sm_103a with plain nvcc (no cmake).

Each translation unit compiles in parallel into ``_build/`` next to the
package, then nvcc links them (static cudart, driver entry points resolved
at run time) into ``matrix_optimizer_step_gb300/libdmuon.so``.  Rebuilds only
what changed (source or shared header newer than the object).
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdmuon.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

SOURCES = ["api.cu", "plan.cu", "step.cu", "host_io.cu", "lpt.cpp", "k_stream.cu", "k_ns_simt.cu", "k_ns_tc.cu", "k_ns_tc2.cu", "noalloc.cu"]
HEADERS = ["internal.h", "runtime.h", "ptx.cuh", "host_util.h", "ns_epilogue.cuh"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags():
    inc = ["-I", os.path.join(ROOT, "include")]
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3,-fvisibility=hidden"] + ARCH + inc


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src, os.path.join(ROOT, "include", "dmuon.h")] + [os.path.join(CSRC, h) for h in HEADERS]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def _compile(nvcc, src, verbose):
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, src + ".o")
    if not _stale(obj, path):
        return obj, None
    cmd = [nvcc] + _flags() + ["-c", path, "-o", obj]
    if src.endswith(".cu") and verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, (r.stdout + r.stderr).strip()


def build(verbose=False, force=False):
    """Compile and link; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    if force:
        for f in os.listdir(BUILD):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD, f))
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s, verbose), SOURCES))
    objs = [o for o, _ in results]
    if verbose:
        for (o, log) in results:
            if log:
                print(f"--- {os.path.basename(o)}\n{log}")
    if (not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs)):
        tmp = LIB + ".tmp"
        cmd = [nvcc, "-shared"] + ARCH + ["-o", tmp] + objs + ["-ldl", "-lpthread", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
