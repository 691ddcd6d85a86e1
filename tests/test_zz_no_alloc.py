"""The allocation-free scan, pr_exclusive_scan_noalloc, through the C ABI.

Some callers must not allocate device memory: code running inside a
framework that owns all device memory through its own pool and hands out
only buffers it has already carved. For them the library offers its
look-back exclusive scan (the step that turns in-degrees into in_ptr) with a
fixed static scratch instead of cudaMalloc. These tests check that it gives
the same offsets as the existing path (pr_graph_create + pr_get_in_csr), on
two calls in a row; that it refuses sizes its scratch cannot hold, negative
counts and totals beyond int32; and, in a fresh process, that its calls take
no device memory.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import os
import subprocess
import sys
import textwrap

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


def test_rejects_a_negative_count_in_a_later_tile(lib):
    counts = np.ones(5 * 4096 + 11, dtype=np.int32)
    counts[3 * 4096 + 5] = -2
    d_counts = torch.from_numpy(counts).cuda()
    d_out = torch.zeros(len(counts) + 1, dtype=torch.int32, device="cuda")
    st = lib.pr_exclusive_scan_noalloc(d_counts.data_ptr(), d_out.data_ptr(), len(counts), None)
    assert st == prg.PR_ERR_INVALID_ARG
    assert "negative" in prg.pr_last_error()
    # the next call, with valid counts, is not affected by the error word
    counts[3 * 4096 + 5] = 2
    got = noalloc_offsets(lib, counts)
    assert np.array_equal(got, np.concatenate([[0], np.cumsum(counts, dtype=np.int64)]))


def test_rejects_a_total_beyond_int32(lib):
    counts = np.full(3 * 4096, 1 << 20, dtype=np.int32)   # total 3 * 2^32 / 1024 > 2^31
    d_counts = torch.from_numpy(counts).cuda()
    d_out = torch.zeros(len(counts) + 1, dtype=torch.int32, device="cuda")
    st = lib.pr_exclusive_scan_noalloc(d_counts.data_ptr(), d_out.data_ptr(), len(counts), None)
    assert st == prg.PR_ERR_TOO_LARGE
    assert "INT32_MAX" in prg.pr_last_error()
    # exactly INT32_MAX is still representable
    counts = np.zeros(2 * 4096 + 3, dtype=np.int32)
    counts[0] = (1 << 30)
    counts[-1] = (1 << 30) - 1
    got = noalloc_offsets(lib, counts)
    assert int(got[-1]) == (1 << 31) - 1


def test_calls_take_no_device_memory_in_a_fresh_process():
    """In a process that has built no graph, the library's pool does not
    exist, and the free device memory the driver reports does not move over
    a series of calls (the first call, which loads the kernels, is left out
    of the comparison)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = textwrap.dedent("""
        import sys
        sys.path.insert(0, %r)
        import numpy as np, torch
        import pagerank_power_iteration_gb300 as prg
        L = prg.lib()
        n = prg.PR_SCAN_NOALLOC_MAX
        counts = torch.ones(n, dtype=torch.int32, device="cuda")
        out = torch.empty(n + 1, dtype=torch.int32, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        assert L.pr_exclusive_scan_noalloc(counts.data_ptr(), out.data_ptr(), 1000, s) == 0
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for k in (n, 12345, n - 1, 0, 1):
            assert L.pr_exclusive_scan_noalloc(counts.data_ptr(), out.data_ptr(), k, s) == 0, prg.pr_last_error()
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert int(out[1]) == 1
        assert prg.pr_test_pool_used_bytes() == 0   # the library's pool was never created
        print("FREE", free0, free1)
        assert free0 == free1, (free0, free1)
    """ % root)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FREE" in r.stdout
