"""Input generators: sizes, structure and determinism (CPU only)."""
import numpy as np
import pytest

import graphgen as gg


def _check_simple(rp, ci, n):
    assert rp[0] == 0 and rp[-1] == len(ci) and np.all(np.diff(rp) >= 0)
    assert ci.min(initial=0) >= 0 and ci.max(initial=0) < n
    src = np.repeat(np.arange(n), np.diff(rp))
    assert not np.any(src == ci), "self-loop"
    for u in range(0, n, max(1, n // 2000)):
        row = ci[rp[u]:rp[u + 1]]
        assert np.all(np.diff(row) > 0), "rows sorted, no duplicates"


def test_citation30k_recipe():
    rp, ci = gg.workload("citation30k")
    n = 30000
    _check_simple(rp, ci, n)
    outdeg = np.diff(rp)
    assert int((outdeg == 0).sum()) == round(0.079 * n)
    assert outdeg[0] == 0  # nobody earlier to cite
    assert outdeg.max() <= 500 and outdeg[3:][outdeg[3:] > 0].min() >= 3
    src = np.repeat(np.arange(n), outdeg)
    assert np.all(ci < src), "a paper cites only earlier papers"
    assert 290_000 <= len(ci) <= 350_000
    indeg = np.bincount(ci, minlength=n)
    assert indeg.max() > 100 * indeg.mean()  # preferential attachment: heavy in-degree tail


def test_rmat_deterministic_across_threads():
    a = gg.rmat(12, seed=7, threads=1)
    b = gg.rmat(12, seed=7, threads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    c = gg.rmat(12, seed=8, threads=4)
    assert not np.array_equal(a[1][:1000], c[1][:1000])


def test_rmat_structure():
    rp, ci = gg.rmat(14, seed=2)
    n = 1 << 14
    _check_simple(rp, ci, n)
    assert 0.85 * 16 * n < len(ci) < 16 * n
    indeg = np.bincount(ci, minlength=n)
    outdeg = np.diff(rp)
    # skew: low ids (many zero bits) are the hubs
    assert indeg[0] > 50 * indeg.mean() and outdeg[0] > 50 * outdeg.mean()
    assert (indeg == 0).mean() > 0.2 and (outdeg == 0).mean() > 0.2


def test_er_recipe_and_determinism():
    n = 20000
    rp, ci = gg.erdos_renyi(n, 16, 0.1, seed=5, threads=3)
    _check_simple(rp, ci, n)
    outdeg = np.diff(rp)
    assert int((outdeg == 0).sum()) == round(0.1 * n)
    assert set(np.unique(outdeg)) == {0, 16}
    rp2, ci2 = gg.erdos_renyi(n, 16, 0.1, seed=5, threads=1)
    assert np.array_equal(ci, ci2)


def test_structured_graphs():
    rp, ci = gg.star_in(5)
    assert list(ci) == [0] * 5 and list(np.diff(rp)) == [0, 1, 1, 1, 1, 1]
    rp, ci = gg.chain(4)
    assert list(ci) == [1, 2, 3] and rp[-2] == rp[-1]
    rp, ci = gg.circulant(5, (1, 2))
    assert list(ci[:2]) == [1, 2] and len(ci) == 10
    rp, ci = gg.single()
    assert list(rp) == [0, 0] and len(ci) == 0
