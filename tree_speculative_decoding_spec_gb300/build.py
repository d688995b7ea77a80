"""Build the spec_tree shared library (libspec_tree.so) in-tree for sm_103a.

Each CUDA translation unit is compiled by nvcc in parallel, then linked into
one shared object next to this file.  Objects go to ``_build/`` at the
repository root (git-ignored).  A unit is rebuilt when it, or any header under
csrc/ or include/, is newer than its object.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libspec_tree.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]:
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime():
    m = 0.0
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".cuh", ".h")):
                m = max(m, os.path.getmtime(os.path.join(d, f)))
    return m


def _compile(nvcc, src, obj, extra):
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, r.returncode, r.stdout + r.stderr, cmd


def build_library(force=False, verbose=False, extra_flags=()):
    """Compile every csrc/*.cu and link libspec_tree.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    hdr = _headers_mtime()
    jobs = []
    objs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr):
            jobs.append((src, obj))
    workers = max(1, min(len(jobs), os.cpu_count() or 4))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            results = list(ex.map(lambda j: _compile(nvcc, j[0], j[1], list(extra_flags)), jobs))
        failed = [r for r in results if r[1] != 0]
        for src, rc, out, cmd in results:
            if verbose or rc != 0:
                sys.stderr.write(f"[nvcc] {os.path.basename(src)} rc={rc}\n{out}")
        if failed:
            raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(f[0]) for f in failed))
    newest = max(os.path.getmtime(o) for o in objs)
    if force or jobs or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        cmd = [nvcc, *ARCH, "-shared", "-o", LIB, *objs, "--cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
