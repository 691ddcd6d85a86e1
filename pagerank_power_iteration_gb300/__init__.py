"""PageRank power iteration on one GB300 GPU (sm_103a): Python binding.

This module marshals arguments into the C ABI declared in
``include/pagerank.h`` (same function names) and adds a small ``Graph``
convenience class over torch tensors. Every step of the computation runs in
the CUDA library ``libpagerank_gb300.so``; there is no CPU fallback. When the
library is missing the first call raises ``PageRankError``; build it with
``pagerank_power_iteration_gb300.build.build()``.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

__all__ = [
    "PR_OK", "PR_NOT_CONVERGED", "PR_ERR_INVALID_ARG", "PR_ERR_INVALID_GRAPH",
    "PR_ERR_TOO_LARGE", "PR_ERR_OOM", "PR_ERR_CUDA", "PR_ERR_TIMEOUT", "PR_F32", "PR_F64",
    "PR_GATHER_LOAD", "PR_GATHER_TMA", "PR_GATHER_BOTH",
    "PageRankError", "pr_graph_info", "pr_run_stats", "lib", "library_path",
    "pr_graph_create", "pr_run", "pr_get_in_csr", "pr_graph_get_info", "pr_graph_last_run",
    "pr_graph_destroy", "pr_last_error", "pr_version", "pr_exclusive_scan_noalloc",
    "pr_measure_gather_rate", "PR_SCAN_NOALLOC_MAX", "PR_LAYOUT_SLACK", "max_edges", "Graph", "EXPORTED_SYMBOLS",
    "pr_test_fail_alloc_after", "pr_test_pool_used_bytes", "pr_test_scan_timeout",
    "pr_options", "pr_graph_create_ex", "PR_BUILD_STAGES", "BUILD_STAGES",
]

PR_OK = 0
PR_NOT_CONVERGED = 1
PR_ERR_INVALID_ARG = -1
PR_ERR_INVALID_GRAPH = -2
PR_ERR_TOO_LARGE = -3
PR_ERR_OOM = -4
PR_ERR_CUDA = -5
PR_ERR_TIMEOUT = -6
PR_F32 = 0
PR_F64 = 1
PR_GATHER_LOAD = 0
PR_GATHER_TMA = 1
PR_GATHER_BOTH = 2

EXPORTED_SYMBOLS = ("pr_graph_create", "pr_graph_create_ex", "pr_run", "pr_get_in_csr", "pr_graph_get_info",
                    "pr_graph_last_run", "pr_graph_destroy", "pr_last_error", "pr_version",
                    "pr_exclusive_scan_noalloc", "pr_measure_gather_rate",
                    # test hooks (include/pagerank_testing.h)
                    "pr_test_fail_alloc_after", "pr_test_pool_used_bytes", "pr_test_scan_timeout")
PR_SCAN_NOALLOC_MAX = 1 << 26
PR_LAYOUT_SLACK = 8192
PR_BUILD_STAGES = 8
BUILD_STAGES = ("degrees", "sources", "sort", "offsets", "order", "layout", "relabel", "finish")


def max_edges(n: int) -> int:
    """Largest m that pr_graph_create accepts for n vertices: m <= 2^31 - 1 and
    m + 3 min(n, m) + PR_LAYOUT_SLACK <= 2^31 - 1 (the padded work layout keeps
    int32 offsets)."""
    cap = (1 << 31) - 1
    best = cap - PR_LAYOUT_SLACK - 3 * n          # when n <= m
    if best >= n:
        return min(cap, best)
    return (cap - PR_LAYOUT_SLACK) // 4           # when m < n: m + 3m <= cap - slack

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpagerank_gb300.so")


class PageRankError(RuntimeError):
    """A negative pr_status from the library, with pr_last_error()'s message."""

    def __init__(self, status: int, message: str):
        super().__init__(f"pagerank error {status}: {message}")
        self.status = status


class pr_options(ctypes.Structure):
    _fields_ = [("thread_max", ctypes.c_int32), ("warp_max", ctypes.c_int32),
                ("stage_timing", ctypes.c_int32)]


class pr_graph_info(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("m", ctypes.c_int64), ("n_dangling", ctypes.c_int64),
                ("rows_zero", ctypes.c_int64), ("rows_thread", ctypes.c_int64),
                ("rows_warp", ctypes.c_int64), ("rows_cta", ctypes.c_int64),
                ("edges_thread", ctypes.c_int64), ("edges_warp", ctypes.c_int64),
                ("edges_cta", ctypes.c_int64), ("cta_chunks", ctypes.c_int64),
                ("cta_chunk_edges", ctypes.c_int32), ("iterate_grid", ctypes.c_int32),
                ("device_bytes", ctypes.c_int64), ("build_launches", ctypes.c_int32),
                ("edges_hot_f32", ctypes.c_int64), ("edges_hot_f64", ctypes.c_int64),
                ("thread_max", ctypes.c_int32), ("warp_max", ctypes.c_int32),
                ("build_ms", ctypes.c_float), ("build_stage_ms", ctypes.c_float * PR_BUILD_STAGES)]

    def as_dict(self):
        d = {k: getattr(self, k) for k, _ in self._fields_}
        d["build_stage_ms"] = dict(zip(BUILD_STAGES, list(self.build_stage_ms)))
        return d


class pr_run_stats(ctypes.Structure):
    _fields_ = [("iterations", ctypes.c_int32), ("converged", ctypes.c_int32),
                ("l1", ctypes.c_double), ("dangling_mass", ctypes.c_double),
                ("loop_ms", ctypes.c_float), ("total_ms", ctypes.c_float),
                ("launches", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded CUDA library (ctypes). Raises PageRankError if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(library_path):
            raise PageRankError(PR_ERR_CUDA, f"CUDA library not built: {library_path} is missing "
                                "(run pagerank_power_iteration_gb300.build.build())")
        L = ctypes.CDLL(library_path)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
        L.pr_graph_create.argtypes = [i64, i64, vp, vp, vp, ctypes.POINTER(vp)]
        L.pr_graph_create.restype = ctypes.c_int
        L.pr_graph_create_ex.argtypes = [i64, i64, vp, vp, ctypes.POINTER(pr_options), vp, ctypes.POINTER(vp)]
        L.pr_graph_create_ex.restype = ctypes.c_int
        L.pr_run.argtypes = [vp, dbl, dbl, i32, ctypes.c_int, vp, vp,
                             ctypes.POINTER(i32), ctypes.POINTER(dbl), vp]
        L.pr_run.restype = ctypes.c_int
        L.pr_get_in_csr.argtypes = [vp, vp, vp, vp]
        L.pr_get_in_csr.restype = ctypes.c_int
        L.pr_graph_get_info.argtypes = [vp, ctypes.POINTER(pr_graph_info)]
        L.pr_graph_get_info.restype = ctypes.c_int
        L.pr_graph_last_run.argtypes = [vp, ctypes.POINTER(pr_run_stats)]
        L.pr_graph_last_run.restype = ctypes.c_int
        L.pr_graph_destroy.argtypes = [vp]
        L.pr_graph_destroy.restype = None
        L.pr_last_error.argtypes = []
        L.pr_last_error.restype = ctypes.c_char_p
        L.pr_version.argtypes = []
        L.pr_version.restype = ctypes.c_char_p
        L.pr_exclusive_scan_noalloc.argtypes = [vp, vp, i64, vp]
        L.pr_exclusive_scan_noalloc.restype = ctypes.c_int
        L.pr_measure_gather_rate.argtypes = [i64, ctypes.c_int, i64, ctypes.c_int, ctypes.POINTER(dbl), vp]
        L.pr_measure_gather_rate.restype = ctypes.c_int
        L.pr_test_fail_alloc_after.argtypes = [i64]
        L.pr_test_fail_alloc_after.restype = None
        L.pr_test_pool_used_bytes.argtypes = [ctypes.POINTER(i64)]
        L.pr_test_pool_used_bytes.restype = ctypes.c_int
        L.pr_test_scan_timeout.argtypes = [i64, i32, vp]
        L.pr_test_scan_timeout.restype = ctypes.c_int
        _lib = L
        return L


# ----------------------------------------------------------- the C ABI, 1:1 --

def pr_graph_create(n: int, m: int, row_ptr: int, col_idx: int, stream: int | None = None) -> int:
    """Raw call: pointers as integers. Returns the handle (an integer)."""
    h = ctypes.c_void_p()
    st = lib().pr_graph_create(n, m, row_ptr, col_idx, stream, ctypes.byref(h))
    _check(st)
    return h.value


def pr_graph_create_ex(n: int, m: int, row_ptr: int, col_idx: int, thread_max: int = 32,
                       warp_max: int = 1024, stage_timing: bool = False, stream: int | None = None) -> int:
    """Raw call with options (class thresholds, per-stage build timing). Returns the handle."""
    opts = pr_options(int(thread_max), int(warp_max), 1 if stage_timing else 0)
    h = ctypes.c_void_p()
    st = lib().pr_graph_create_ex(n, m, row_ptr, col_idx, ctypes.byref(opts), stream, ctypes.byref(h))
    _check(st)
    return h.value


def pr_run(graph: int, d: float, tol: float, max_iter: int, dtype: int, ranks_out: int,
           x_init: int | None = None, stream: int | None = None):
    """Raw call. Returns (status, iterations, l1); status is PR_OK or PR_NOT_CONVERGED."""
    it = ctypes.c_int32(0)
    l1 = ctypes.c_double(0.0)
    st = lib().pr_run(graph, d, tol, max_iter, dtype, ranks_out, x_init,
                      ctypes.byref(it), ctypes.byref(l1), stream)
    _check(st)
    return st, it.value, l1.value


def pr_get_in_csr(graph: int, in_ptr: int, in_col: int, stream: int | None = None) -> None:
    _check(lib().pr_get_in_csr(graph, in_ptr, in_col, stream))


def pr_graph_get_info(graph: int) -> dict:
    info = pr_graph_info()
    _check(lib().pr_graph_get_info(graph, ctypes.byref(info)))
    return info.as_dict()


def pr_graph_last_run(graph: int) -> dict:
    stats = pr_run_stats()
    _check(lib().pr_graph_last_run(graph, ctypes.byref(stats)))
    return stats.as_dict()


def pr_graph_destroy(graph: int) -> None:
    if graph:
        lib().pr_graph_destroy(graph)


def pr_exclusive_scan_noalloc(counts: int, offsets: int, count: int, stream: int | None = None) -> None:
    """Raw call: device pointers as integers. offsets[i] = sum of counts[:i], i in [0, count].

    Allocates no device memory (static scratch for up to PR_SCAN_NOALLOC_MAX
    elements, shared by all calls: do not overlap calls on the GPU)."""
    _check(lib().pr_exclusive_scan_noalloc(counts, offsets, count, stream))


def pr_measure_gather_rate(n: int, dtype: int, gathers: int, stream: int | None = None,
                           path: int = PR_GATHER_LOAD) -> float:
    """Raw call. Random gathers per second from an n-element state vector of
    dtype (PR_F32 or PR_F64) on the current GPU, through `path`
    (PR_GATHER_LOAD: the warps' loads, the ceiling of the update's gathers that
    shared memory does not serve; PR_GATHER_TMA: TMA tile::gather4 copies;
    PR_GATHER_BOTH: both at once)."""
    rate = ctypes.c_double(0.0)
    _check(lib().pr_measure_gather_rate(n, dtype, gathers, path, ctypes.byref(rate), stream))
    return rate.value


def pr_test_fail_alloc_after(k: int) -> None:
    """Test hook: the k-th pool allocation from now fails with PR_ERR_OOM (0: off)."""
    lib().pr_test_fail_alloc_after(int(k))


def pr_test_pool_used_bytes() -> int:
    """Test hook: bytes of the current device's library pool in use (0 if no pool yet)."""
    used = ctypes.c_int64(0)
    _check(lib().pr_test_pool_used_bytes(ctypes.byref(used)))
    return used.value


def pr_test_scan_timeout(count: int, spin_limit: int, stream: int | None = None) -> int:
    """Test hook: a scan whose first tile never publishes. Returns the status
    (PR_ERR_TIMEOUT when the bounded look-back waits ran out) without raising."""
    return lib().pr_test_scan_timeout(int(count), int(spin_limit), stream)


def pr_last_error() -> str:
    return lib().pr_last_error().decode()


def pr_version() -> str:
    return lib().pr_version().decode()


def _check(st: int) -> None:
    if st < 0:
        raise PageRankError(st, pr_last_error())


# ----------------------------------------------------------- convenience ---

def _ptr(a) -> int | None:
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be contiguous")
        return a.ctypes.data
    if not a.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return a.data_ptr()


def _check_vector(a, n: int, dtype, name: str, device: int) -> None:
    """Raises unless ``a`` (numpy array or torch tensor) holds exactly n
    contiguous values of ``dtype`` (torch.float32 or torch.float64), in host
    memory or on CUDA device ``device``."""
    import torch
    if isinstance(a, np.ndarray):
        want = np.float32 if dtype == torch.float32 else np.float64
        if a.dtype != want:
            raise TypeError(f"{name} must be {np.dtype(want).name}, got {a.dtype}")
        size, contiguous = a.size, a.flags["C_CONTIGUOUS"]
    elif isinstance(a, torch.Tensor):
        if a.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {a.dtype}")
        # host memory, or memory of the graph's own GPU: a kernel must never
        # be handed another GPU's memory
        if a.device.type != "cpu" and a.device != torch.device("cuda", device):
            raise ValueError(f"{name} must be on the CPU or on cuda:{device}, got {a.device}")
        size, contiguous = a.numel(), a.is_contiguous()
    else:
        raise TypeError(f"{name} must be a numpy array or a torch tensor")
    if size != n:
        raise ValueError(f"{name} must hold n = {n} values, got {size}")
    if not contiguous:
        raise ValueError(f"{name} must be contiguous")


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Graph:
    """A graph resident on the current CUDA device.

    ``row_ptr`` (int64[n+1]) and ``col_idx`` (int32[m]) form the out-edge CSR;
    they may be numpy arrays or torch tensors, on the host or on the device.
    ``thread_max`` and ``warp_max`` are the in-degree class thresholds, and
    ``stage_timing`` records the build's stages (``info()["build_stage_ms"]``).
    """

    def __init__(self, row_ptr, col_idx, stream=None, thread_max: int = 32, warp_max: int = 1024,
                 stage_timing: bool = False):
        import torch
        if isinstance(row_ptr, np.ndarray):
            row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
            col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
        else:
            if row_ptr.dtype != torch.int64 or col_idx.dtype != torch.int32:
                raise TypeError("row_ptr must be int64 and col_idx int32")
            row_ptr = row_ptr.contiguous()
            col_idx = col_idx.contiguous()
        self.n = int(row_ptr.shape[0]) - 1
        self.m = int(col_idx.shape[0])
        self.device = torch.cuda.current_device()
        self._h = pr_graph_create_ex(self.n, self.m, _ptr(row_ptr), _ptr(col_idx) if self.m else None,
                                     thread_max, warp_max, stage_timing, _stream(stream))

    @property
    def handle(self) -> int:
        return self._h

    def run(self, d: float = 0.85, tol: float = 1e-6, max_iter: int = 200, dtype=None,
            out=None, x_init=None, stream=None):
        """Runs the power iteration. Returns (ranks, iterations, l1, converged).

        ``ranks`` is ``out`` if given (host or device tensor/array of ``dtype``)
        or a new CUDA tensor. ``converged`` is False when tol > 0 and
        max_iter updates did not reach L1 < tol. ``x_init`` (warm start) must
        be a probability vector: non-negative, summing to 1.
        """
        import torch
        dtype = torch.float32 if dtype is None else dtype
        if dtype not in (torch.float32, torch.float64):
            raise TypeError("dtype must be torch.float32 or torch.float64")
        code = PR_F32 if dtype == torch.float32 else PR_F64
        if out is None:
            out = torch.empty(self.n, dtype=dtype, device=f"cuda:{self.device}")
        # the library reads and writes exactly n values of the run's type
        # through these pointers, so a shorter buffer or another type would be
        # read or written out of bounds
        _check_vector(out, self.n, dtype, "out", self.device)
        if x_init is not None:
            _check_vector(x_init, self.n, dtype, "x_init", self.device)
        st, it, l1 = pr_run(self._h, float(d), float(tol), int(max_iter), code, _ptr(out),
                            _ptr(x_init), _stream(stream))
        return out, it, l1, st == PR_OK

    def in_csr(self, stream=None):
        """The in-edge CSR as host numpy arrays (in_ptr int32[n+1], in_col int32[m])."""
        in_ptr = np.empty(self.n + 1, dtype=np.int32)
        in_col = np.empty(max(self.m, 1), dtype=np.int32)
        pr_get_in_csr(self._h, in_ptr.ctypes.data, in_col.ctypes.data, _stream(stream))
        return in_ptr, in_col[: self.m]

    def info(self) -> dict:
        return pr_graph_get_info(self._h)

    def last_run(self) -> dict:
        return pr_graph_last_run(self._h)

    def close(self) -> None:
        h, self._h = getattr(self, "_h", None), None
        if h:
            pr_graph_destroy(h)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
