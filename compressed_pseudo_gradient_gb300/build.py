"""Builds libspl.so (the codec's CUDA kernels and C ABI) in-tree for sm_103a with nvcc.

Each translation unit compiles in parallel; the result is linked with the static CUDA runtime
into ``compressed_pseudo_gradient_gb300/libspl.so``.  The same sources compiled with
``-DSPL_CHECKED=1`` give ``libspl_checked.so``, a diagnostic build whose kernels test every
memory index before the access (recording, not trapping, a bad one; see include/spl_checked.h).
Rebuilds only when a source or header is newer than the libraries.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libspl.so")
CHECKED_LIB_PATH = os.path.join(PKG, "libspl_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
    # every floating-point step of the codec is an explicit round-to-nearest intrinsic;
    # keep the compiler from contracting anything else and keep IEEE division/denormals
    "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspl.so")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) +
            [os.path.abspath(__file__)])


def is_stale() -> bool:
    for lib in (LIB_PATH, CHECKED_LIB_PATH):
        if not os.path.exists(lib):
            return True
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(p) > t for p in _deps()):
            return True
    return False


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libspl.so and libspl_checked.so if stale (or when forced); returns the
    path of libspl.so."""
    if not force and not is_stale():
        return LIB_PATH
    cc = nvcc()
    variants = [(LIB_PATH, BUILD_DIR, []),
                (CHECKED_LIB_PATH, os.path.join(BUILD_DIR, "checked"), ["-DSPL_CHECKED=1"])]
    procs = []
    objs = {lib: [] for lib, _, _ in variants}
    for lib, odir, extra in variants:
        os.makedirs(odir, exist_ok=True)
        for src in _sources():
            obj = os.path.join(odir, os.path.basename(src)[:-3] + ".o")
            cmd = [cc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
            objs[lib].append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            print(out, end="")
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {', '.join(os.path.basename(f) for f in failed)}")
    for lib, _, _ in variants:
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs[lib]],
                       check=True)
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
