"""The multi-core CPU baseline (OpenMP pull) that bench.py times beside the
GPU path computes the same thing as the oracle: the same in-edge CSR bit for
bit, and the same ranks (to fp64 rounding) at the same number of updates,
whatever the thread count."""
import numpy as np
import pytest

import cpu_parallel
import graphgen as gg
import oracle
from gpu_util import F64, assert_ranks_close

D = 0.85


@pytest.fixture(scope="module", autouse=True)
def built():
    oracle.build()
    cpu_parallel.build()


GRAPHS = {
    "rmat14": lambda: gg.rmat(14, seed=6),
    "citation": lambda: gg.citation(n=4000, seed=3),
    "star_in": lambda: gg.star_in(3000),
    "dups_loops": lambda: gg.random_sparse(2000, 20000, seed=11, dangling_frac=0.3),
    "no_edges": lambda: gg.from_edges(7, [], []),
}


@pytest.mark.parametrize("name", sorted(GRAPHS))
@pytest.mark.parametrize("threads", [1, 4])
def test_transpose_matches_the_oracle(name, threads):
    rp, ci = GRAPHS[name]()
    ip, ic = cpu_parallel.transpose(rp, ci, threads=threads)
    oip, oic = oracle.transpose(rp, ci)
    assert np.array_equal(ip, oip)
    assert np.array_equal(ic, oic)


@pytest.mark.parametrize("name", sorted(GRAPHS))
@pytest.mark.parametrize("threads", [1, 4])
def test_ranks_match_the_oracle(name, threads):
    rp, ci = GRAPHS[name]()
    r = cpu_parallel.pagerank(rp, ci, D, tol=1e-10, max_iter=300, threads=threads)
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=r["iters"])
    assert_ranks_close(r["x"], ref["x"], F64, f"{name} threads={threads}")
    refc = oracle.pagerank(rp, ci, D, tol=1e-10, max_iter=300)
    assert abs(refc["iters"] - r["iters"]) <= 1
    assert abs(r["x"].sum() - 1.0) <= F64["sum"]


def test_fixed_updates_and_invalid_input():
    rp, ci = gg.rmat(10, seed=1)
    r = cpu_parallel.pagerank(rp, ci, D, tol=0.0, max_iter=5, threads=2)
    assert r["iters"] == 5 and r["status"] == cpu_parallel.OK
    bad = ci.copy()
    bad[0] = len(rp) + 3
    with pytest.raises(ValueError):
        cpu_parallel.transpose(rp, bad, threads=2)
