"""Build the CUDA library in-tree for sm_103a (GB300).

    python -m gradient_ring_all_gb300.build [--force] [--verbose-ptxas] [--checked]

Compiles each csrc/*.cu into _build/*.o in parallel with nvcc and links
lib/libgradient_ring_all.so against the shared CUDA runtime.  A stamp of the
sources and flags skips the work when nothing changed.  --checked builds the
bounds-checked library instead (RA_CHECKED=1: every kernel verifies each
global range it touches and reports a violation through the error word),
into _build_checked/ and lib/libgradient_ring_all_checked.so; the tests use
it, the product does not.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libgradient_ring_all.so")
LIB_CHECKED = os.path.join(LIBDIR, "libgradient_ring_all_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build gradient_ring_all_gb300")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    deps = sorted(f for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    return cu, deps


def _stamp(extra) -> str:
    h = hashlib.sha256()
    cu, deps = _sources()
    for f in cu + deps:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    with open(os.path.join(ROOT, "include", "ring_allreduce.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool | None = None) -> str:
    if checked is None:  # the library the binding will load
        checked = os.environ.get("GRADIENT_RING_ALL_CHECKED") == "1"
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if checked:
        extra.append("-DRA_CHECKED=1")
    bdir = BUILD + "_checked" if checked else BUILD
    lib = LIB_CHECKED if checked else LIB
    stamp_file = os.path.join(bdir, "stamp")
    stamp = _stamp(extra)
    if not force and os.path.exists(lib) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return lib
    nvcc = _nvcc()
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cu, _ = _sources()

    def compile_one(f):
        obj = os.path.join(bdir, f[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, f), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (f, r.stdout, r.stderr))
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(len(cu), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, cu))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + ".tmp%d" % os.getpid()
    libdir = _cuda_lib_dir(nvcc)
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for o, _ in results],
           "-Xlinker", "-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv,
                checked=True if "--checked" in sys.argv else None))
