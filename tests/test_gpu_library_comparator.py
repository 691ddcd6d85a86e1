"""The library-composed comparator that bench.py times beside the CUDA path
(a library sort for the transpose, a cuSPARSE CSR SpMV per update, torch
elementwise ops and reductions for the rest) computes the same power
iteration: its ranks match the oracle's at the same number of updates, and
its converged update count is within one of the oracle's."""
import numpy as np
import pytest

import graphgen as gg
import oracle
from gpu_util import F32, F64, assert_ranks_close

torch = pytest.importorskip("torch")
import bench  # noqa: E402

pytestmark = pytest.mark.gpu
D = 0.85


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    oracle.build()


@pytest.mark.parametrize("name,dtype", [("rmat14", "f32"), ("citation", "f32"), ("rmat14", "f64")])
def test_library_comparator_matches_the_oracle(name, dtype):
    rp, ci = gg.rmat(14, seed=6) if name == "rmat14" else gg.citation(n=5000, seed=3)
    tt = {"f32": torch.float32, "f64": torch.float64}[dtype]
    x, ups, _, _ = bench.library_pagerank(rp, ci, D, 1e-6, 200, tt, torch.device("cuda:0"))
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=ups)
    assert_ranks_close(x.cpu().numpy(), ref["x"], F32 if dtype == "f32" else F64, f"{name} {dtype}")
    refc = oracle.pagerank(rp, ci, D, tol=1e-6, max_iter=200)
    assert abs(refc["iters"] - ups) <= 1


def test_library_comparator_fixed_updates():
    rp, ci = gg.rmat(12, seed=2)
    x, ups, _, _ = bench.library_pagerank(rp, ci, D, 0.0, 200, torch.float32, torch.device("cuda:0"), fixed=7)
    assert ups == 7
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=7)
    assert_ranks_close(x.cpu().numpy(), ref["x"], F32, "fixed 7")
