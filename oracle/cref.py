"""ctypes access to oracle/mean_ref.c (the rank-ordered average in plain C,
single-threaded and split over threads).

TEST INFRASTRUCTURE ONLY, like the rest of oracle/: used by its pin test and
by the benchmark's CPU-baseline leg for timing context.  build() returns the
path of the compiled library, or None when no C compiler is available (the
C oracle is optional; the numpy oracle is the definition the tests use).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "mean_ref.c")
LIB = os.path.join(_HERE, "libmean_ref.so")
_lib = None


def build():
    """Compile mean_ref.c (with OpenMP when the compiler has it); returns the
    library path, or None if it cannot be built here."""
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    base = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", SRC, "-o", LIB]
    for extra in (["-fopenmp"], []):
        try:
            r = subprocess.run(base + extra, capture_output=True, text=True, timeout=120)
        except (OSError, subprocess.TimeoutExpired):
            return None
        if r.returncode == 0:
            return LIB
    return None


def _load():
    global _lib
    if _lib is None:
        path = build()
        if path is None:
            return None
        lib = ctypes.CDLL(path)
        for name in ("oracle_grad_mean_f32", "oracle_grad_mean_f32_threads"):
            getattr(lib, name).argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]
            getattr(lib, name).restype = None
        lib.oracle_threads.restype = ctypes.c_int32
        _lib = lib
    return _lib


def available() -> bool:
    return _load() is not None


def threads() -> int:
    return int(_load().oracle_threads())


def grad_mean_c(grads, threaded: bool = False) -> np.ndarray:
    """The average of fp32 arrays, computed by the C oracle."""
    lib = _load()
    arrs = [np.ascontiguousarray(g, dtype=np.float32).reshape(-1) for g in grads]
    n = len(arrs)
    ptrs = (ctypes.c_void_p * n)(*[a.ctypes.data for a in arrs])
    out = np.empty(arrs[0].size, np.float32)
    fn = lib.oracle_grad_mean_f32_threads if threaded else lib.oracle_grad_mean_f32
    fn(ctypes.addressof(ptrs), n, out.size, out.ctypes.data)
    return out
