"""Builds libspd.so (all CUDA sources, sm_103a) in-tree with nvcc.

Each ``csrc/*.cu`` compiles to an object in ``_build/`` (in parallel), then
the objects link into ``libspd.so`` next to this file with the CUDA runtime
linked statically.  A stamp of the sources and flags skips up-to-date builds.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import re
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libspd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspd.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


# sources of the sparse/dense attention call per K/V cache type (planner
# kernels and that cache type's tensor-core attention kernel): what a
# DRAM-traffic capture of that call depends on
_PLAN_SOURCES = ("dispatch.cu", "plan.cu", "plan.cuh", "spd_internal.cuh", "tc_ptx.cuh", "tmap.cuh")
ATTENTION_SOURCES = {"e4m3": ("attention_e4m3_rows_tc.cu", "attention_tc.cu") + _PLAN_SOURCES,
                     "bf16": ("attention_bf16_tc.cu",) + _PLAN_SOURCES}


def _code_only(text: bytes) -> bytes:
    """C/C++ source without its comments and blank-line differences: what
    the compiler sees, so a comment edit does not change a kernel stamp."""
    t = text.decode("utf-8", errors="replace")
    t = re.sub(r"/\*.*?\*/", " ", t, flags=re.S)
    t = re.sub(r"//[^\n]*", "", t)
    lines = [ln.rstrip() for ln in t.splitlines()]
    return "\n".join(ln for ln in lines if ln).encode()


def _stamp(names=None) -> str:
    """Hash of the sources (all of them, or -- comments stripped -- the named
    files of csrc) and the compiler flags."""
    h = hashlib.sha256()
    paths = (sorted(glob.glob(os.path.join(CSRC, "*")) + [os.path.join(INCLUDE, "spd.h")]) if names is None
             else [os.path.join(CSRC, n) for n in sorted(names)])
    for path in paths:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode())
            h.update(f.read() if names is None else _code_only(f.read()))
    # flags with the checkout's own paths made relative: the same sources
    # stamp the same on every machine
    flags = [os.path.relpath(f, ROOT) if f.startswith(ROOT) else f for f in ARCH + NVCC_FLAGS]
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libspd.so; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    stamp_path = os.path.join(BUILD_DIR, "stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read() == stamp:
                return LIB_PATH
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose:
        for _, log in results:
            print(log)
    objs = [o for o, _ in results]
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "--cudart", "static", "-o", tmp, *objs, "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link of libspd.so failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB_PATH)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return LIB_PATH


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
