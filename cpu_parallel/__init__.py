"""Multi-core CPU PageRank (OpenMP pull over the in-edge CSR), a measured
baseline that bench.py times beside the GPU path on all host cores.

Neither the oracle nor the product: the CUDA library never imports or calls
it, and the three share no code. The arithmetic lives in ``pagerank_omp.c``;
this module compiles it with the host C compiler (``-fopenmp``) and marshals
numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagerank_omp.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpagerank_omp.so")

OK = 0
NOT_CONVERGED = 1
ERR_ARG = -1
ERR_GRAPH = -2
ERR_OOM = -4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles ``pagerank_omp.c`` into ``cpu_parallel/_build/libpagerank_omp.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O3", "-fopenmp", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                   check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            l = ctypes.CDLL(build())
            i64, i32, f64, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
            l.po_transpose.argtypes = [i64, i64, p, p, ctypes.c_int, p, p]
            l.po_transpose.restype = ctypes.c_int
            l.po_pagerank.argtypes = [i64, i64, p, p, f64, f64, i32, ctypes.c_int, p, p, p, p, p]
            l.po_pagerank.restype = ctypes.c_int
            l.po_max_threads.argtypes = []
            l.po_max_threads.restype = ctypes.c_int
            _lib = l
        return _lib


def max_threads() -> int:
    return int(lib().po_max_threads())


def _csr(row_ptr, col_idx):
    return (np.ascontiguousarray(row_ptr, dtype=np.int64), np.ascontiguousarray(col_idx, dtype=np.int32))


def transpose(row_ptr, col_idx, threads: int | None = None):
    """In-edge CSR (in_ptr int64[n+1], in_col int32[m])."""
    rp, ci = _csr(row_ptr, col_idx)
    n, m = len(rp) - 1, len(ci)
    in_ptr = np.empty(n + 1, dtype=np.int64)
    in_col = np.empty(max(m, 1), dtype=np.int32)
    st = lib().po_transpose(n, m, rp.ctypes.data, ci.ctypes.data, threads or max_threads(),
                            in_ptr.ctypes.data, in_col.ctypes.data)
    if st != OK:
        raise ValueError(f"po_transpose failed with status {st}")
    return in_ptr, in_col[:m]


def pagerank(row_ptr, col_idx, d: float = 0.85, tol: float = 1e-6, max_iter: int = 200,
             threads: int | None = None) -> dict:
    """Ranks (fp64) and run figures: iters, l1, status, t_transpose, t_loop (s), threads."""
    rp, ci = _csr(row_ptr, col_idx)
    n, m = len(rp) - 1, len(ci)
    th = threads or max_threads()
    x = np.empty(n, dtype=np.float64)
    it, l1 = ctypes.c_int32(0), ctypes.c_double(0.0)
    tt, tl = ctypes.c_double(0.0), ctypes.c_double(0.0)
    st = lib().po_pagerank(n, m, rp.ctypes.data, ci.ctypes.data, d, tol, max_iter, th, x.ctypes.data,
                           ctypes.byref(it), ctypes.byref(l1), ctypes.byref(tt), ctypes.byref(tl))
    if st < 0:
        raise ValueError(f"po_pagerank failed with status {st}")
    return {"x": x, "iters": it.value, "l1": l1.value, "status": st, "t_transpose": tt.value,
            "t_loop": tl.value, "threads": th}
