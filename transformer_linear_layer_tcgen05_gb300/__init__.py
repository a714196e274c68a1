"""GB300 (sm_103a) forward linear-layer family: matmul, matmul_residual,
matmul_residual_swiglu_a and their binary16-weight variants.

The compute path is the C-ABI library ``liblin.so`` (``include/lin.h``),
built by ``build.build_library()``; ``lin`` is its thin ctypes binding and
``workloads`` the seeded synthetic inputs. Importing this package loads
nothing: the library is opened on first use and a missing library is an
error, never a fallback.
"""

__all__ = ["lin", "workloads", "build"]
