"""Build libtwell.so in-tree for sm_103a (nvcc, one translation unit per kernel
family, compiled in parallel, then linked into one shared library), and the
benchmark's row-gather probe as a library of its own (libtwell_probe.so)."""
from __future__ import annotations

import concurrent.futures
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libtwell.so")
PROBE_LIB = os.path.join(OUT_DIR, "libtwell_probe.so")
# the checked (debug) build: every index a gather reads is bounds-checked on
# the device and reported as TWELL_ERR_INDEX (see common.cuh)
CHECKED_LIB = os.path.join(OUT_DIR, "libtwell_checked.so")

SOURCES = ["api.cu", "gemm_tc.cu", "gate_smallm.cu", "pack.cu", "sparse_fwd.cu", "sparse_bwd.cu",
           "selftest.cu"]
PROBE_SOURCES = ["gather_probe.cu"]
HEADERS = ["common.cuh", "ell_gather.cuh", "gemm_tc.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _newest_input() -> float:
    files = [os.path.join(CSRC, s) for s in SOURCES + PROBE_SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "twell.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build_checked(force: bool = False) -> str:
    """Compile and link libtwell_checked.so (-DTWELL_CHECKED) if any input is
    newer than it."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(CHECKED_LIB) and os.path.getmtime(CHECKED_LIB) >= _newest_input():
        return CHECKED_LIB
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + "_checked.o")
        cmd = [nvcc] + NVCC_FLAGS + ["-DTWELL_CHECKED", "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, res.stdout, res.stderr))
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = CHECKED_LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (res.stdout, res.stderr))
    os.replace(tmp, CHECKED_LIB)
    return CHECKED_LIB


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libtwell.so and libtwell_probe.so if any input is
    newer than them."""
    os.makedirs(OUT_DIR, exist_ok=True)
    newest = _newest_input()
    if (not force and all(os.path.exists(p) and os.path.getmtime(p) >= newest
                          for p in (LIB, PROBE_LIB))):
        return LIB
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, res.stdout, res.stderr))
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    srcs = SOURCES + PROBE_SOURCES
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = dict(zip(srcs, ex.map(compile_one, srcs)))
    for lib, group in ((LIB, SOURCES), (PROBE_LIB, PROBE_SOURCES)):
        tmp = lib + ".tmp%d" % os.getpid()
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + [objs[g] for g in group]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n%s%s" % (res.stdout, res.stderr))
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    if "--checked" in sys.argv:
        print(build_checked(force=True))
    else:
        print(build(force=True, verbose="-v" in sys.argv))
