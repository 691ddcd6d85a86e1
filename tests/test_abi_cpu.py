"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
symbol include/pagerank.h declares, and rejects bad scalar arguments on the
host before touching CUDA. No compute call is made here."""
import ctypes
import os
import re

import pytest

import pagerank_power_iteration_gb300 as prg
from pagerank_power_iteration_gb300 import build as prbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    """Every function the headers under include/ declare."""
    text = ""
    for name in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if name.endswith(".h"):
            with open(os.path.join(ROOT, "include", name)) as f:
                text += f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pr_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    prbuild.build()
    return prg.lib()


def test_header_declares_the_abi():
    assert header_functions() == sorted(prg.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(L):
    for name in header_functions():
        assert hasattr(L, name), name


def test_only_the_abi_is_exported(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", prg.library_path], capture_output=True,
                         text=True, check=True).stdout
    syms = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert syms == set(prg.EXPORTED_SYMBOLS)


def test_built_for_sm_103a():
    with open(os.path.join(os.path.dirname(prg.__file__), "_build", "iterate.cu.ptxas.txt")) as f:
        assert "sm_103a" in f.read()


def test_version_and_error_strings(L):
    assert "sm_103a" in prg.pr_version()
    assert isinstance(prg.pr_last_error(), str)


@pytest.mark.parametrize("n,m,code", [(0, 0, prg.PR_ERR_INVALID_ARG), (-3, 0, prg.PR_ERR_INVALID_ARG),
                                      (5, -1, prg.PR_ERR_INVALID_ARG),
                                      (1 << 31, 0, prg.PR_ERR_TOO_LARGE),
                                      (10, 1 << 31, prg.PR_ERR_TOO_LARGE)])
def test_create_rejects_bad_sizes_on_host(L, n, m, code):
    rp = (ctypes.c_int64 * 2)(0, 0)
    h = ctypes.c_void_p()
    st = L.pr_graph_create(n, m, ctypes.addressof(rp), None, None, ctypes.byref(h))
    assert st == code and not h.value
    assert prg.pr_last_error()


def test_create_rejects_null_pointers_on_host(L):
    h = ctypes.c_void_p()
    assert L.pr_graph_create(4, 0, None, None, None, ctypes.byref(h)) == prg.PR_ERR_INVALID_ARG
    rp = (ctypes.c_int64 * 5)(0, 1, 2, 3, 4)
    assert L.pr_graph_create(4, 4, ctypes.addressof(rp), None, None, ctypes.byref(h)) == prg.PR_ERR_INVALID_ARG
    assert L.pr_graph_create(4, 0, ctypes.addressof(rp), None, None, None) == prg.PR_ERR_INVALID_ARG


@pytest.mark.parametrize("d,tol,max_iter,dtype", [(1.5, 1e-6, 10, 0), (-0.1, 1e-6, 10, 0),
                                                  (float("nan"), 1e-6, 10, 0),
                                                  (0.85, float("nan"), 10, 0), (0.85, 1e-6, 0, 0),
                                                  (0.85, 1e-6, 10, 7)])
def test_run_rejects_bad_arguments_on_host(L, d, tol, max_iter, dtype):
    out = (ctypes.c_float * 4)()
    # a NULL graph is reported first; the scalar checks are exercised with a
    # fake non-NULL handle that is never dereferenced because they fail first
    assert L.pr_run(None, 0.85, 1e-6, 10, 0, ctypes.addressof(out), None, None, None, None) == prg.PR_ERR_INVALID_ARG
    fake = ctypes.c_void_p(ctypes.addressof(out))
    st = L.pr_run(fake, d, tol, max_iter, dtype, ctypes.addressof(out), None, None, None, None)
    assert st == prg.PR_ERR_INVALID_ARG


@pytest.mark.parametrize("n,dtype,gathers", [(0, 0, 1024), (-5, 0, 1024), ((1 << 31) - 1, 0, 1024),
                                              (1000, 0, 0), (1000, 0, (1 << 30) + 1), (1000, 7, 1024)])
def test_gather_rate_rejects_bad_arguments_on_host(L, n, dtype, gathers):
    rate = ctypes.c_double(0.0)
    assert L.pr_measure_gather_rate(1000, 0, 1024, prg.PR_GATHER_LOAD, None, None) == prg.PR_ERR_INVALID_ARG
    st = L.pr_measure_gather_rate(n, dtype, gathers, prg.PR_GATHER_LOAD, ctypes.byref(rate), None)
    assert st == prg.PR_ERR_INVALID_ARG
    assert rate.value == 0.0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(prg, "_lib", None)
    monkeypatch.setattr(prg, "library_path", str(tmp_path / "nope.so"))
    with pytest.raises(prg.PageRankError):
        prg.lib()


def test_create_rejects_graphs_whose_padded_layout_overflows(L):
    # m + 3 min(n, m) + PR_LAYOUT_SLACK must fit in int32 (checked on the host,
    # before any device work or dereference of the inputs)
    rp = (ctypes.c_int64 * 2)(0, 0)
    ci = (ctypes.c_int32 * 1)(0)
    h = ctypes.c_void_p()
    for n in (1 << 24, 1000, (1 << 31) - 2):
        m = prg.max_edges(n) + 1
        st = L.pr_graph_create(n, m, ctypes.addressof(rp), ctypes.addressof(ci), None, ctypes.byref(h))
        assert st == prg.PR_ERR_TOO_LARGE and not h.value, (n, m)
        assert "int32" in prg.pr_last_error()
    # the limit itself: every extra edge past max_edges(n) breaks the bound
    for n in (1 << 24, 1000, (1 << 31) - 2):
        m = prg.max_edges(n)
        assert m + 3 * min(n, m) + prg.PR_LAYOUT_SLACK <= (1 << 31) - 1
        m1 = m + 1
        assert m1 + 3 * min(n, m1) + prg.PR_LAYOUT_SLACK > (1 << 31) - 1 or m1 > (1 << 31) - 1


def test_layout_slack_matches_the_header():
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(prg.__file__)), "include", "pagerank.h")).read()
    assert int(re.search(r"#define PR_LAYOUT_SLACK (\d+)", hdr).group(1)) == prg.PR_LAYOUT_SLACK


def test_run_rejects_mismatched_buffers_before_calling_the_library(monkeypatch):
    # pr_run reads x_init and writes the ranks through raw pointers, n values of
    # the run's type, so the binding must refuse any other buffer before the call
    torch = pytest.importorskip("torch")
    import numpy as np
    g = prg.Graph.__new__(prg.Graph)        # no device handle: nothing may reach the library
    g.n, g.m, g.device, g._h = 10, 0, 0, None
    calls = []
    monkeypatch.setattr(prg, "pr_run", lambda *a: calls.append(a))
    good = np.zeros(10, dtype=np.float32)
    cases = [
        dict(out=np.zeros(9, dtype=np.float32)),                 # too short
        dict(out=np.zeros(11, dtype=np.float32)),                # too long
        dict(out=np.zeros(10, dtype=np.float64)),                # fp64 buffer, fp32 run
        dict(out=torch.zeros(10, dtype=torch.float64)),
        dict(out=np.zeros(20, dtype=np.float32)[::2]),           # not contiguous
        dict(out=[0.0] * 10),                                    # not an array
        dict(out=good, x_init=np.zeros(9, dtype=np.float32)),
        dict(out=good, x_init=torch.zeros(10, dtype=torch.float64)),
        dict(out=good, x_init=np.zeros(10, dtype=np.float64)),
        dict(out=np.zeros(10, dtype=np.float32), dtype=torch.float64),
        dict(out=good, dtype=torch.int32),
        # neither host memory nor the graph's GPU (a meta tensor stands in for
        # another device here, where no GPU exists)
        dict(out=torch.zeros(10, dtype=torch.float32, device="meta")),
        dict(out=good, x_init=torch.zeros(10, dtype=torch.float32, device="meta")),
    ]
    for kw in cases:
        with pytest.raises((TypeError, ValueError)):
            g.run(0.85, 1e-6, 10, **kw)
    assert not calls


def test_gather_rate_rejects_an_unknown_path_on_host(L):
    rate = ctypes.c_double(0.0)
    for n, dtype, gathers, path in ((0, 0, 10, 1), (10, 2, 10, 2), (10, 0, 0, 1), (10, 0, 10, 3), (10, 0, 10, -1)):
        st = L.pr_measure_gather_rate(n, dtype, gathers, path, ctypes.byref(rate), None)
        assert st == prg.PR_ERR_INVALID_ARG, (n, dtype, gathers, path)


@pytest.mark.parametrize("thread_max,warp_max", [(0, 1024), (33, 1024), (-1, 5), (32, 31), (8, 7),
                                                 (8, -5), (32, 8193), (1, 1 << 20)])
def test_create_ex_rejects_bad_options_on_host(L, thread_max, warp_max):
    opts = prg.pr_options(thread_max, warp_max, 0)
    h = ctypes.c_void_p()
    st = L.pr_graph_create_ex(10, 0, None, None, ctypes.byref(opts), None, ctypes.byref(h))
    assert st == prg.PR_ERR_INVALID_ARG
    assert ("thread_max" in prg.pr_last_error()) or ("warp_max" in prg.pr_last_error())
    assert h.value is None


def test_options_struct_matches_the_header():
    hdr = open(os.path.join(ROOT, "include", "pagerank.h")).read()
    assert "#define PR_OPTIONS_DEFAULT {32, 1024, 0}" in hdr
    assert int(re.search(r"#define PR_BUILD_STAGES (\d+)", hdr).group(1)) == prg.PR_BUILD_STAGES
    assert [f for f, _ in prg.pr_options._fields_] == ["thread_max", "warp_max", "stage_timing"]
