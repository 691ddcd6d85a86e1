"""Seeded synthetic directed graphs as out-edge CSR (row_ptr int64[n+1], col_idx int32[m]).

Input generation only: nothing here computes any part of PageRank. The tests
of the CUDA library and of the oracle both take their inputs from this module.

Large generators (RMAT, Erdos-Renyi, citation-like) are in ``graphgen.c`` and
are compiled on first use with the host C compiler; the small structured
graphs with closed-form PageRank (cycles, stars, chains, ...) are built here in
numpy.

Named workloads (``workload(name)``) follow the graph shapes the PageRank pages
measure:

=============  =====================================================================
name           recipe
=============  =====================================================================
citation30k    n = 30,000, seed 1; 7.9 % dangling; out-degree ~ k^-2.1 on [3, 500];
               targets by preferential attachment (in-degree so far + 1)
rmat18         RMAT scale 18, edge factor 16, a/b/c/d = .57/.19/.19/.05, seed 2
rmat22         RMAT scale 22, same parameters, seed 3
rmat24         RMAT scale 24, same parameters, seed 4
er24           n = 2^24, 10 % dangling, out-degree 16 uniform distinct targets, seed 5
=============  =====================================================================
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "graphgen.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgraphgen.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles ``graphgen.c`` (gcc -O2 -fopenmp) into ``graphgen/_build``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu99", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, dbl, u64, vp = (ctypes.c_int64, ctypes.c_int32, ctypes.c_double,
                                  ctypes.c_uint64, ctypes.c_void_p)
        lib.gg_rmat.argtypes = [i32, i64, dbl, dbl, dbl, u64, i32, vp, vp, vp]
        lib.gg_rmat.restype = ctypes.c_int
        lib.gg_er.argtypes = [i64, i32, dbl, u64, i32, vp, vp, vp]
        lib.gg_er.restype = ctypes.c_int
        lib.gg_citation.argtypes = [i64, dbl, i32, i32, dbl, u64, vp, vp, i64, vp]
        lib.gg_citation.restype = ctypes.c_int
        _lib = lib
        return lib


def _vp(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _threads(threads):
    return int(threads) if threads else (os.cpu_count() or 1)


def rmat(scale: int, edge_factor: int = 16, a: float = 0.57, b: float = 0.19, c: float = 0.19,
         seed: int = 2, threads: int | None = None):
    """RMAT digraph, 2^scale vertices, edge_factor * 2^scale draws, deduplicated, no self-loops."""
    n = 1 << scale
    cap = edge_factor * n
    row_ptr = np.empty(n + 1, dtype=np.int64)
    col_idx = np.empty(max(cap, 1), dtype=np.int32)
    m = ctypes.c_int64(0)
    rc = _load().gg_rmat(scale, edge_factor, a, b, c, seed, _threads(threads),
                         _vp(row_ptr), _vp(col_idx), ctypes.byref(m))
    if rc != 0:
        raise RuntimeError(f"gg_rmat failed ({rc})")
    return row_ptr, col_idx[: m.value]


def erdos_renyi(n: int, deg: int = 16, dangling_frac: float = 0.1, seed: int = 5,
                threads: int | None = None):
    """Every non-dangling vertex gets `deg` distinct uniform targets other than itself."""
    row_ptr = np.empty(n + 1, dtype=np.int64)
    col_idx = np.empty(max(n * deg, 1), dtype=np.int32)
    m = ctypes.c_int64(0)
    rc = _load().gg_er(n, deg, dangling_frac, seed, _threads(threads), _vp(row_ptr),
                       _vp(col_idx), ctypes.byref(m))
    if rc != 0:
        raise RuntimeError(f"gg_er failed ({rc})")
    return row_ptr, col_idx[: m.value]


def citation(n: int = 30000, zipf_s: float = 2.1, kmin: int = 3, kmax: int = 500,
             dangling_frac: float = 0.079, seed: int = 1):
    """Citation-like digraph: power-law out-degrees, preferential-attachment targets."""
    row_ptr = np.empty(n + 1, dtype=np.int64)
    cap = n * min(kmax, n - 1)
    col_idx = np.empty(max(cap, 1), dtype=np.int32)
    m = ctypes.c_int64(0)
    rc = _load().gg_citation(n, zipf_s, kmin, kmax, dangling_frac, seed, _vp(row_ptr),
                             _vp(col_idx), cap, ctypes.byref(m))
    if rc != 0:
        raise RuntimeError(f"gg_citation failed ({rc})")
    return row_ptr, col_idx[: m.value].copy()


WORKLOADS = {
    "citation30k": dict(kind="citation", n=30000, seed=1),
    "rmat18": dict(kind="rmat", scale=18, seed=2),
    "rmat22": dict(kind="rmat", scale=22, seed=3),
    "rmat24": dict(kind="rmat", scale=24, seed=4),
    "er24": dict(kind="er", n=1 << 24, seed=5),
}


def workload(name: str, threads: int | None = None):
    """Returns the out-edge CSR of a named workload (see the module docstring)."""
    w = WORKLOADS[name]
    if w["kind"] == "citation":
        return citation(n=w["n"], seed=w["seed"])
    if w["kind"] == "rmat":
        return rmat(w["scale"], 16, 0.57, 0.19, 0.19, seed=w["seed"], threads=threads)
    if w["kind"] == "er":
        return erdos_renyi(w["n"], 16, 0.1, seed=w["seed"], threads=threads)
    raise KeyError(name)


# --------------------------------------------------------------------------
# small structured graphs (numpy), and CSR assembly from an edge list
# --------------------------------------------------------------------------

def from_edges(n: int, src, dst):
    """Out-edge CSR from an edge list; rows keep the list's order (stable by source)."""
    src = np.asarray(src, dtype=np.int64)
    dst = np.asarray(dst, dtype=np.int64)
    order = np.argsort(src, kind="stable")
    counts = np.bincount(src, minlength=n) if src.size else np.zeros(n, dtype=np.int64)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    return row_ptr, dst[order].astype(np.int32)


def single(self_loop: bool = False):
    """One vertex; with self_loop it has the edge 0 -> 0."""
    return from_edges(1, [0] if self_loop else [], [0] if self_loop else [])


def cycle(n: int):
    """Directed cycle 0 -> 1 -> ... -> n-1 -> 0."""
    u = np.arange(n)
    return from_edges(n, u, (u + 1) % n)


def circulant(n: int, offsets=(1, 2)):
    """u -> u + k (mod n) for every k in offsets."""
    u = np.arange(n)
    src = np.concatenate([u for _ in offsets])
    dst = np.concatenate([(u + k) % n for k in offsets])
    return from_edges(n, src, dst)


def star_in(k: int):
    """k leaves 1..k each with one edge to the centre 0 (the centre is dangling)."""
    leaves = np.arange(1, k + 1)
    return from_edges(k + 1, leaves, np.zeros(k, dtype=np.int64))


def star_out(k: int):
    """Centre 0 with an edge to each of the k leaves (the leaves are dangling)."""
    leaves = np.arange(1, k + 1)
    return from_edges(k + 1, np.zeros(k, dtype=np.int64), leaves)


def chain(n: int):
    """0 -> 1 -> ... -> n-1 (the last vertex is dangling)."""
    u = np.arange(n - 1)
    return from_edges(n, u, u + 1)


def random_digraph(n: int, p: float, dangling_frac: float = 0.0, seed: int = 0,
                   self_loops: bool = False, multi: bool = False):
    """Bernoulli(p) digraph on n vertices with a chosen fraction forced dangling.

    With ``multi`` some edges are listed twice; with ``self_loops`` u -> u may appear.
    """
    rng = np.random.default_rng(seed)
    a = rng.random((n, n)) < p
    if not self_loops:
        np.fill_diagonal(a, False)
    k = int(round(dangling_frac * n))
    if k:
        a[rng.choice(n, size=k, replace=False), :] = False
    src, dst = np.nonzero(a)
    if multi and src.size:
        extra = rng.random(src.size) < 0.3
        src = np.concatenate([src, src[extra]])
        dst = np.concatenate([dst, dst[extra]])
    return from_edges(n, src, dst)


def random_sparse(n: int, m: int, seed: int = 0, dangling_frac: float = 0.0):
    """m uniform random edges (duplicates and self-loops allowed) among n vertices."""
    rng = np.random.default_rng(seed)
    src = rng.integers(0, n, size=m)
    dst = rng.integers(0, n, size=m)
    k = int(round(dangling_frac * n))
    if k:
        dead = np.zeros(n, dtype=bool)
        dead[rng.choice(n, size=k, replace=False)] = True
        keep = ~dead[src]
        src, dst = src[keep], dst[keep]
    return from_edges(n, src, dst)
