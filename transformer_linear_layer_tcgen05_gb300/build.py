"""Build ``liblin.so`` (the C-ABI library of include/lin.h) in-tree with nvcc.

Every translation unit is compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), in parallel, then linked as a
shared library next to this file. Object files go to ``_build/`` at the
repository root. A rebuild happens only when a source or header is newer than
the library.

``build_library(checked=True)`` builds the same sources with
``-DLIN_DEVICE_CHECKS=1`` into ``liblin_checked.so`` (objects in
``_build/checked/``): the checked build, whose kernels check their shared
memory, TMEM, TMA-coordinate and global indices (include/lin.h).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "liblin.so")
CHECKED_LIB_PATH = os.path.join(PKG_DIR, "liblin_checked.so")

SOURCES = ["lin_api.cu", "lin_kernels_tf32.cu", "lin_kernels_f16.cu",
           "lin_kernels_cluster_swiglu.cu", "lin_kernels_cluster_cvt.cu",
           "lin_kernels_cluster_bt.cu", "lin_kernels_cluster_dual.cu", "lin_loss.cu",
           "lin_noalloc.cu", "lin_host.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build liblin.so")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "lin.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(checked: bool = False) -> bool:
    lib = CHECKED_LIB_PATH if checked else LIB_PATH
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False, extra_flags=(),
                  checked: bool = False) -> str:
    """Compile and link liblin.so (or, ``checked``, liblin_checked.so); return
    its path. Raises on any failure."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    if not force and up_to_date(checked):
        return lib_path
    nvcc = _nvcc()
    build_dir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    if checked:
        extra_flags = (*extra_flags, "-DLIN_DEVICE_CHECKS=1")
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH, *CFLAGS, *extra_flags, *os.environ.get("LIN_NVCC_FLAGS", "").split(),
               "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            print(out, file=sys.stderr)
        if p.returncode != 0:
            failed.append(f"{src}:\n{out}")
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib_path + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    if verbose:
        print(" ".join(link), file=sys.stderr)
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv,
                        checked="--checked" in sys.argv))
