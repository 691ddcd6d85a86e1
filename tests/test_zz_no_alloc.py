"""The allocation-free scan, pr_exclusive_scan_noalloc, through the C ABI.

Some callers must not allocate device memory: a framework that owns all
device memory through its own pool, or work issued while another thread
captures a CUDA graph in global capture mode. For them the library offers its
look-back exclusive scan (the step that turns in-degrees into in_ptr) with a
fixed static scratch instead of cudaMalloc. These tests check that it gives
the same offsets as the existing path (pr_graph_create + pr_get_in_csr), on
two calls in a row, and that it refuses sizes its scratch cannot hold.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import graphgen as gg

torch = pytest.importorskip("torch")
import pagerank_power_iteration_gb300 as prg  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from pagerank_power_iteration_gb300 import build
    build.build()
    return prg.lib()


def existing_offsets(rp, ci):
    """in_ptr as the existing entry points produce it."""
    with prg.Graph(rp, ci) as g:
        in_ptr, _ = g.in_csr()
    return in_ptr


def noalloc_offsets(lib, counts):
    d_counts = torch.from_numpy(np.ascontiguousarray(counts, dtype=np.int32)).cuda()
    d_out = torch.full((len(counts) + 1,), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.pr_exclusive_scan_noalloc(d_counts.data_ptr(), d_out.data_ptr(), len(counts), stream)
    assert st == prg.PR_OK, prg.pr_last_error()
    return d_out.cpu().numpy()


def test_matches_the_existing_entry_point_on_two_calls_in_a_row(lib):
    # two graphs of different sizes (many tiles, ragged last tile), one call each
    for rp, ci in (gg.workload("rmat18"), gg.citation(n=30000, seed=1)):
        ref = existing_offsets(rp, ci)
        counts = np.diff(ref.astype(np.int64)).astype(np.int32)
        got = noalloc_offsets(lib, counts)
        assert np.array_equal(got, ref)


def test_repeated_calls_do_not_depend_on_earlier_contents(lib):
    # the scratch keeps the previous call's contents; each call clears what it uses
    rng = np.random.default_rng(5)
    big = rng.integers(0, 40, size=3 * 4096 * 16 + 17).astype(np.int32)
    small = rng.integers(0, 9, size=1000).astype(np.int32)
    for counts in (big, small, big):
        got = noalloc_offsets(lib, counts)
        ref = np.concatenate([[0], np.cumsum(counts, dtype=np.int64)])
        assert np.array_equal(got, ref)


def test_empty_input(lib):
    assert np.array_equal(noalloc_offsets(lib, np.zeros(0, dtype=np.int32)), [0])


def test_rejects_sizes_beyond_the_static_scratch(lib):
    d = torch.zeros(8, dtype=torch.int32, device="cuda")
    st = lib.pr_exclusive_scan_noalloc(d.data_ptr(), d.data_ptr(), prg.PR_SCAN_NOALLOC_MAX + 1, None)
    assert st == prg.PR_ERR_TOO_LARGE
    assert "static scratch" in prg.pr_last_error()
    st = lib.pr_exclusive_scan_noalloc(d.data_ptr(), d.data_ptr(), -1, None)
    assert st == prg.PR_ERR_INVALID_ARG


def test_rejects_host_pointers(lib):
    host = np.zeros(8, dtype=np.int32)
    d = torch.zeros(9, dtype=torch.int32, device="cuda")
    st = lib.pr_exclusive_scan_noalloc(host.ctypes.data, d.data_ptr(), 8, None)
    assert st == prg.PR_ERR_INVALID_ARG
