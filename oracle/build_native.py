"""Compile the oracle's C contraction (``gemm_f64.c``) into a shared library.

TEST INFRASTRUCTURE ONLY: part of the oracle. ``lin_oracle`` calls
``build()`` on first use; the package's ``build()`` entry point runs this file
as a script so that the checker is compiled with everything else. Plain gcc,
no target-specific flags, and no contraction of a*b+c into a fused
multiply-add (``-ffp-contract=off``), so that the x86 and Arm hosts round
every step alike. OpenMP shares rows between threads where the compiler has
it; without it the loop runs on one thread and computes the same bits.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "gemm_f64.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libgemm_f64.so")
BASE_FLAGS = ["-O3", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def _cc() -> str:
    for cand in (os.environ.get("CC"), shutil.which("gcc"), shutil.which("cc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("no C compiler (gcc) found: the oracle's contraction is C")


def up_to_date() -> bool:
    return (os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(SOURCE),
                                                  os.path.getmtime(os.path.abspath(__file__))))


def build(force: bool = False) -> str:
    """Compile when stale; return the library's path. Raises on failure."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = _cc()
    # A private temporary name, then an atomic rename: processes that build
    # at once never load a half-written file.
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=OUT_DIR)
    os.close(fd)
    try:
        last = ""
        for extra in (["-fopenmp"], []):
            r = subprocess.run([cc, *BASE_FLAGS, *extra, SOURCE, "-o", tmp, "-lm"],
                               stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
            if r.returncode == 0:
                os.replace(tmp, LIB_PATH)
                return LIB_PATH
            last = r.stdout
        raise RuntimeError("oracle C build failed:\n" + last)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
