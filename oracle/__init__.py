"""PageRank oracle: a plain single-threaded fp64 CPU implementation.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package. The product path
(``pagerank_power_iteration_gb300``) never imports, links or calls it, and the
two share no code.

The arithmetic lives in ``pagerank_oracle.c`` (see its header for what it
computes and which passage each step follows). This module only compiles that
file with the host C compiler and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagerank_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

OK = 0
NOT_CONVERGED = 1
ERR_ARG = -1
ERR_GRAPH = -2
ERR_OOM = -4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles the oracle into ``oracle/_build/liboracle.so`` (plain gcc, -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
        lib.oracle_check_csr.argtypes = [i64, i64, vp, vp]
        lib.oracle_check_csr.restype = ctypes.c_int
        lib.oracle_transpose.argtypes = [i64, i64, vp, vp, vp, vp]
        lib.oracle_transpose.restype = ctypes.c_int
        lib.oracle_pagerank.argtypes = [i64, i64, vp, vp, dbl, dbl, i32, i32,
                                        vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_pagerank.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _csr(row_ptr, col_idx):
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    n = row_ptr.shape[0] - 1
    return n, col_idx.shape[0], row_ptr, col_idx


class OracleError(RuntimeError):
    pass


def check_csr(row_ptr, col_idx) -> int:
    n, m, rp, ci = _csr(row_ptr, col_idx)
    if n < 1:
        return ERR_ARG
    return _load().oracle_check_csr(n, m, _ptr(rp), _ptr(ci))


def transpose(row_ptr, col_idx):
    """Counting-sort transpose. Returns (in_ptr int64[n+1], in_col int32[m])."""
    n, m, rp, ci = _csr(row_ptr, col_idx)
    in_ptr = np.empty(max(n, 0) + 1, dtype=np.int64)
    in_col = np.empty(max(m, 1), dtype=np.int32)
    rc = _load().oracle_transpose(n, m, _ptr(rp), _ptr(ci), _ptr(in_ptr), _ptr(in_col))
    if rc < 0:
        raise OracleError(f"oracle_transpose failed with code {rc}")
    return in_ptr, in_col[:m]


def pagerank(row_ptr, col_idx, d: float = 0.85, tol: float = 1e-6, max_iter: int = 200,
             drop_dangling: bool = False, x_init=None, logs: bool = False):
    """Power iteration in fp64.

    Returns a dict with ``x`` (float64[n]), ``iters``, ``l1``, ``status`` and,
    when ``logs`` is set, per-update ``sum``, ``dmass`` and ``l1_log`` arrays.
    """
    n, m, rp, ci = _csr(row_ptr, col_idx)
    if n < 1:
        raise OracleError("n must be >= 1")
    x = np.empty(n, dtype=np.float64)
    xi = None if x_init is None else np.ascontiguousarray(x_init, dtype=np.float64)
    iters = ctypes.c_int32(0)
    l1 = ctypes.c_double(0.0)
    sl = dl = ll = None
    if logs:
        sl = np.zeros(max_iter, dtype=np.float64)
        dl = np.zeros(max_iter, dtype=np.float64)
        ll = np.zeros(max_iter, dtype=np.float64)
    rc = _load().oracle_pagerank(n, m, _ptr(rp), _ptr(ci), float(d), float(tol),
                                 int(max_iter), int(bool(drop_dangling)), _ptr(xi),
                                 _ptr(x), ctypes.byref(iters), ctypes.byref(l1),
                                 _ptr(sl), _ptr(dl), _ptr(ll))
    if rc < 0:
        raise OracleError(f"oracle_pagerank failed with code {rc}")
    out = {"x": x, "iters": int(iters.value), "l1": float(l1.value), "status": int(rc)}
    if logs:
        k = int(iters.value)
        out["sum"], out["dmass"], out["l1_log"] = sl[:k], dl[:k], ll[:k]
    return out
