"""Parity at the full sizes of the benchmark workloads, in the launch
configuration bench.py times (graph built from a device-resident CSR, fp32,
d = 0.85, tol 1e-6, at most 200 updates).

- The transpose is compared bit for bit with the oracle's counting sort.
- Every rank after 3 fixed updates is compared with the oracle.
- The converged run: iteration count within one update of the oracle's,
  |sum - 1| <= 1e-5, L1 below the tolerance, and ranks within tolerance of
  the oracle rerun for the same number of updates.
- RMAT scale 22 also runs in its fixed-50 mode (tol = 0, exactly 50 updates,
  the timed mode of Day 40's "Results"): every rank against the oracle after
  the same 50 updates, and |sum - 1| <= 1e-5.
- ER at 2^24 also runs in fp64.

Each case takes tens of seconds (the oracle is single-threaded).
"""
import numpy as np
import pytest

import graphgen as gg
import oracle
from gpu_util import F32, F64, assert_ranks_close

torch = pytest.importorskip("torch")
import pagerank_power_iteration_gb300 as prg  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
D = 0.85


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from pagerank_power_iteration_gb300 import build
    build.build()
    oracle.build()


@pytest.fixture(scope="module", params=["rmat22", "rmat24", "er24"])
def workload(request):
    rp, ci = gg.workload(request.param)
    return request.param, rp, ci


def test_full_size_transpose_bit_exact(workload):
    name, rp, ci = workload
    g = prg.Graph(torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda())
    try:
        ip, ic = g.in_csr()
    finally:
        g.close()
    oip, oic = oracle.transpose(rp, ci)
    assert np.array_equal(ip.astype(np.int64), oip), name
    assert np.array_equal(ic, oic), name


def test_full_size_fixed_updates(workload):
    name, rp, ci = workload
    g = prg.Graph(torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda())
    try:
        x, it, l1, _ = g.run(D, 0.0, 3)
        x = x.cpu().numpy()
    finally:
        g.close()
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=3)
    assert it == 3
    assert_ranks_close(x, ref["x"], F32, f"{name} after 3 updates")


def test_full_size_converged(workload):
    name, rp, ci = workload
    g = prg.Graph(torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda())
    try:
        x, it, l1, conv = g.run(D, 1e-6, 200)
        x = x.cpu().numpy()
    finally:
        g.close()
    assert conv and l1 < 1e-6
    assert abs(x.astype(np.float64).sum() - 1.0) <= F32["sum"]
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=it)
    assert_ranks_close(x, ref["x"], F32, f"{name} after {it} updates")
    refc = oracle.pagerank(rp, ci, D, tol=1e-6, max_iter=200)
    assert abs(refc["iters"] - it) <= 1, (refc["iters"], it)


def test_rmat22_fixed_50_updates():
    rp, ci = gg.workload("rmat22")
    g = prg.Graph(torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda())
    try:
        x, it, l1, conv = g.run(D, 0.0, 50)
        x = x.cpu().numpy()
    finally:
        g.close()
    assert it == 50 and conv   # tol <= 0: exactly max_iter updates, reported as success
    assert abs(x.astype(np.float64).sum() - 1.0) <= F32["sum"]
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=50)
    assert ref["iters"] == 50
    assert_ranks_close(x, ref["x"], F32, "rmat22 after 50 fixed updates")
    # the L1 of the 50th update, against the oracle's (fp32 terms: 2% or 4 ulp(1))
    assert abs(l1 - ref["l1"]) <= max(0.02 * ref["l1"], 4 * 2.0 ** -23), (l1, ref["l1"])


def test_er24_fp64():
    rp, ci = gg.workload("er24")
    g = prg.Graph(torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda())
    try:
        x, it, l1, conv = g.run(D, 1e-10, 200, dtype=torch.float64)
        x = x.cpu().numpy()
    finally:
        g.close()
    assert conv and l1 < 1e-10
    assert abs(x.sum() - 1.0) <= F64["sum"]
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=it)
    assert_ranks_close(x, ref["x"], F64, f"er24 fp64 after {it} updates")
