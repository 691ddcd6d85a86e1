"""Pins that tie the oracle to what the pages and mathematics fix, not to itself.

Each test is chosen so that a plausible slip in the oracle (a dropped
dangling term, D/n outside the d*(...) bracket, a transposed adjacency, a
wrong divisor, a wrong stopping rule) fails at least one of them. The planted
-mistake test at the end checks exactly that, on the CPU, by editing a copy
of the oracle's C source.
"""
import os
import subprocess
import ctypes
import tempfile

import numpy as np
import pytest

import graphgen as gg
import oracle
from conftest import day40_case, read_golden, simple_dataset_11, tiny6

D = 0.85


# ---------------------------------------------------------------- helpers ---

def dense_google(row_ptr, col_idx, d):
    """Dense fp64 Google matrix, built independently of the oracle:
    P[v, u] = (#edges u->v) / outdeg(u); a dangling column is 1/n everywhere;
    G = d P + (1 - d)/n * 1 1^T (column-stochastic)."""
    n = len(row_ptr) - 1
    P = np.zeros((n, n))
    outdeg = np.diff(row_ptr)
    for u in range(n):
        if outdeg[u] == 0:
            P[:, u] = 1.0 / n
        else:
            for j in range(row_ptr[u], row_ptr[u + 1]):
                P[col_idx[j], u] += 1.0 / outdeg[u]
    return d * P + (1.0 - d) / n * np.ones((n, n)), P


def solve_fixed_point(row_ptr, col_idx, d):
    """Textbook linear solve of (I - d P) x = (1 - d)/n 1 (numpy.linalg.solve)."""
    n = len(row_ptr) - 1
    _, P = dense_google(row_ptr, col_idx, d)
    return np.linalg.solve(np.eye(n) - d * P, np.full(n, (1.0 - d) / n))


def small_graphs():
    out = [("tiny6", tiny6()), ("simple11", simple_dataset_11()), ("single", gg.single()),
           ("single_loop", gg.single(True)), ("cycle7", gg.cycle(7)),
           ("star_in9", gg.star_in(9)), ("star_out9", gg.star_out(9)), ("chain12", gg.chain(12))]
    for i, frac in enumerate([0.0, 0.1, 0.3, 0.6, 1.0]):
        out.append((f"rand_{frac}", gg.random_digraph(40, 0.12, frac, seed=10 + i)))
    out.append(("rand_multi_loops", gg.random_digraph(48, 0.1, 0.2, seed=99, self_loops=True, multi=True)))
    out.append(("rand64", gg.random_digraph(64, 0.05, 0.25, seed=7)))
    return out


# --------------------------------------------------------- transpose pins ---

def lexsort_transpose(row_ptr, col_idx):
    """Independent transpose: numpy lexsort of (destination, source) pairs."""
    n = len(row_ptr) - 1
    src = np.repeat(np.arange(n), np.diff(row_ptr))
    dst = np.asarray(col_idx, dtype=np.int64)
    order = np.lexsort((src, dst))
    in_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(dst, minlength=n), out=in_ptr[1:])
    return in_ptr, src[order].astype(np.int32)


@pytest.mark.parametrize("name,graph", small_graphs() + [
    ("random_sparse_dups", gg.random_sparse(500, 4000, seed=3, dangling_frac=0.2)),
    ("star_in_big", gg.star_in(3000)),
    ("star_out_big", gg.star_out(3000)),
])
def test_transpose_matches_lexsort(built_oracle, name, graph):
    rp, ci = graph
    ip, ic = oracle.transpose(rp, ci)
    ip2, ic2 = lexsort_transpose(rp, ci)
    assert np.array_equal(ip, ip2)
    assert np.array_equal(ic, ic2)
    assert ip[-1] == len(ci)


def test_transpose_generated_graphs(built_oracle):
    for rp, ci in [gg.citation(n=3000, seed=3), gg.rmat(12, seed=9), gg.erdos_renyi(5000, 16, 0.1, seed=4)]:
        ip, ic = oracle.transpose(rp, ci)
        ip2, ic2 = lexsort_transpose(rp, ci)
        assert np.array_equal(ip, ip2) and np.array_equal(ic, ic2)


def test_transpose_twice_is_identity_on_sorted_rows(built_oracle):
    rp, ci = gg.random_sparse(300, 2500, seed=5)
    # sort each input row so the round trip is well defined
    ci = ci.copy()
    for u in range(300):
        ci[rp[u]:rp[u + 1]].sort()
    ip, ic = oracle.transpose(rp, ci)
    rp2, ci2 = oracle.transpose(ip, ic)
    assert np.array_equal(rp2, rp) and np.array_equal(ci2, ci)


def test_check_csr_rejects_bad_graphs(built_oracle):
    rp, ci = tiny6()
    assert oracle.check_csr(rp, ci) == oracle.OK
    bad = ci.copy(); bad[0] = 6
    assert oracle.check_csr(rp, bad) == oracle.ERR_GRAPH
    bad = ci.copy(); bad[0] = -1
    assert oracle.check_csr(rp, bad) == oracle.ERR_GRAPH
    rbad = rp.copy(); rbad[2], rbad[3] = rbad[3], rbad[2]
    assert oracle.check_csr(rbad, ci) == oracle.ERR_GRAPH
    rbad = rp.copy(); rbad[0] = 1
    assert oracle.check_csr(rbad, ci) == oracle.ERR_GRAPH


# ---------------------------------------------------- dense brute force pins --

@pytest.mark.parametrize("name,graph", small_graphs())
def test_power_iteration_matches_dense_google_matrix(built_oracle, name, graph):
    """k fixed updates agree with k products by the dense Google matrix."""
    rp, ci = graph
    n = len(rp) - 1
    G, _ = dense_google(rp, ci, D)
    x = np.full(n, 1.0 / n)
    for k in (1, 2, 5, 30):
        out = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=k)
        y = x.copy()
        for _ in range(k):
            y = G @ y
        assert out["iters"] == k
        np.testing.assert_allclose(out["x"], y, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("name,graph", small_graphs())
def test_converged_matches_linear_solve(built_oracle, name, graph):
    """The converged iterate solves (I - dP) x = (1-d)/n 1 within the L1 tolerance
    (error <= tol * d / (1 - d) in L1)."""
    rp, ci = graph
    tol = 1e-13
    out = oracle.pagerank(rp, ci, D, tol=tol, max_iter=2000)
    assert out["status"] == oracle.OK
    xs = solve_fixed_point(rp, ci, D)
    assert np.abs(out["x"] - xs).sum() <= tol * D / (1 - D) + 1e-14


@pytest.mark.parametrize("d", [0.0, 0.5, 0.85, 0.99, 1.0])
def test_damping_extremes_against_dense(built_oracle, d):
    rp, ci = gg.random_digraph(30, 0.15, 0.2, seed=21)
    n = 30
    G, _ = dense_google(rp, ci, d)
    y = np.full(n, 1.0 / n)
    for _ in range(12):
        y = G @ y
    out = oracle.pagerank(rp, ci, d, tol=0.0, max_iter=12)
    np.testing.assert_allclose(out["x"], y, rtol=1e-13, atol=1e-15)


def test_x_init_is_the_start_vector(built_oracle):
    rp, ci = gg.random_digraph(25, 0.2, 0.2, seed=4)
    G, _ = dense_google(rp, ci, D)
    rng = np.random.default_rng(1)
    x0 = rng.random(25); x0 /= x0.sum()
    out = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=3, x_init=x0)
    np.testing.assert_allclose(out["x"], G @ (G @ (G @ x0)), rtol=1e-13, atol=1e-16)


# ------------------------------------------------------------- invariants --

@pytest.mark.parametrize("name", ["tiny", "dangling", "star", "chain"])
def test_sum_to_one_after_every_update(built_oracle, name):
    """Day 40, 'One iteration, three shapes of work': the ranks sum to 1 after
    every pass (constant term 1-d, SpMV term d(S-D), dangling term dD)."""
    rp, ci = day40_case(name)
    out = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=100, logs=True)
    assert np.all(np.abs(out["sum"] - 1.0) <= 1e-12)


def test_sum_to_one_on_citation_graph(built_oracle):
    rp, ci = gg.citation(n=30000, seed=1)
    out = oracle.pagerank(rp, ci, D, tol=1e-6, max_iter=200, logs=True)
    assert out["status"] == oracle.OK
    assert np.all(np.abs(out["sum"] - 1.0) <= 1e-12)
    assert out["l1"] < 1e-6 and out["l1_log"][-2] >= 1e-6


def test_stop_rule_is_first_update_below_tol(built_oracle):
    rp, ci = gg.random_digraph(50, 0.1, 0.2, seed=8)
    out = oracle.pagerank(rp, ci, D, tol=1e-9, max_iter=500, logs=True)
    ll = out["l1_log"]
    assert ll[-1] < 1e-9 and np.all(ll[:-1] >= 1e-9)
    assert out["iters"] == len(ll)
    capped = oracle.pagerank(rp, ci, D, tol=1e-9, max_iter=3)
    assert capped["status"] == oracle.NOT_CONVERGED and capped["iters"] == 3


# --------------------------------------------- the dropped dangling term ---

@pytest.mark.parametrize("name", ["tiny", "dangling", "star", "chain"])
def test_dropping_dangling_term_gives_one_minus_dD(built_oracle, name):
    """Day 40: without the redistribution the next total is 1 - d*D."""
    rp, ci = day40_case(name)
    out = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=1, drop_dangling=True, logs=True)
    n = len(rp) - 1
    # summing n doubles in order: rounding error up to about n * eps
    assert abs(out["sum"][0] - (1.0 - D * out["dmass"][0])) <= max(1e-14, n * 2.3e-16)


def test_dropping_dangling_fixed_point_total_and_proportionality(built_oracle):
    """Day 40 'Solution': the broken total settles at S = 1 - D d/(1-d) and the
    broken vector is the correct one times (1-d)/(1-d+d D_correct)."""
    rp, ci = tiny6()
    good = oracle.pagerank(rp, ci, D, tol=1e-15, max_iter=5000, logs=True)
    bad = oracle.pagerank(rp, ci, D, tol=1e-15, max_iter=5000, drop_dangling=True, logs=True)
    dm_bad = bad["dmass"][-1]
    assert abs(bad["x"].sum() - (1.0 - dm_bad * D / (1.0 - D))) <= 1e-12
    dm_good = good["dmass"][-1]
    ratio = bad["x"] / good["x"]
    np.testing.assert_allclose(ratio, (1 - D) / (1 - D + D * dm_good), rtol=1e-11)
    # ranking unchanged
    assert np.array_equal(np.argsort(bad["x"], kind="stable"), np.argsort(good["x"], kind="stable"))


def test_no_dangling_means_drop_has_no_effect(built_oracle):
    rp, ci = day40_case("nodangling")
    a = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=10)
    b = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=10, drop_dangling=True)
    assert np.array_equal(a["x"], b["x"])


# ------------------------------------------------------------ closed forms --

@pytest.mark.parametrize("n", [1, 2, 3, 1000, 65537])
def test_directed_cycle_is_uniform_in_one_update(built_oracle, n):
    rp, ci = gg.cycle(n) if n > 1 else gg.single(True)
    out = oracle.pagerank(rp, ci, D, tol=1e-6, max_iter=200)
    assert out["iters"] == 1
    np.testing.assert_allclose(out["x"], 1.0 / n, rtol=1e-14)


def test_circulant_nodangling_is_uniform(built_oracle):
    rp, ci = day40_case("nodangling")
    out = oracle.pagerank(rp, ci, D, tol=1e-6, max_iter=200)
    assert out["iters"] == 1
    np.testing.assert_allclose(out["x"], 1.0 / 4096, rtol=1e-14)


@pytest.mark.parametrize("k", [1, 5, 10000])
def test_star_leaves_to_centre(built_oracle, k):
    """Fixed point of the update on a star whose k leaves point at a dangling
    centre: x_c = (1 + k d)/(1 + k + k d), leaves (1 - x_c)/k."""
    rp, ci = gg.star_in(k)
    out = oracle.pagerank(rp, ci, D, tol=1e-15, max_iter=1000)
    xc = (1 + k * D) / (1 + k + k * D)
    # the centre sums k leaf terms in order: rounding up to about k * eps
    assert abs(out["x"][0] - xc) <= max(1e-14, k * 2.3e-16)
    np.testing.assert_allclose(out["x"][1:], (1 - xc) / k, rtol=1e-11)
    if k == 10000:
        assert abs(xc - 0.459489) < 1e-6


@pytest.mark.parametrize("k", [1, 7, 10000])
def test_star_centre_to_leaves(built_oracle, k):
    """Centre with k out-edges to dangling leaves: x_c = 1/(n + d), n = k + 1."""
    rp, ci = gg.star_out(k)
    n = k + 1
    out = oracle.pagerank(rp, ci, D, tol=1e-15, max_iter=1000)
    xc = 1.0 / (n + D)
    assert abs(out["x"][0] - xc) <= 1e-14
    np.testing.assert_allclose(out["x"][1:], (1 - xc) / k, rtol=1e-11)


@pytest.mark.parametrize("n", [2, 3, 50, 8192])
def test_chain(built_oracle, n):
    """0 -> 1 -> ... -> n-1: x_i = c (1 - d^(i+1))/(1 - d),
    c = (1 - d)/(n - d (1 - d^n)/(1 - d))."""
    rp, ci = gg.chain(n)
    out = oracle.pagerank(rp, ci, D, tol=1e-14, max_iter=5000)
    c = (1 - D) / (n - D * (1 - D ** n) / (1 - D))
    i = np.arange(n)
    expect = c * (1 - D ** (i + 1)) / (1 - D)
    np.testing.assert_allclose(out["x"], expect, rtol=1e-10, atol=1e-16)


def test_single_node(built_oracle):
    for loop in (False, True):
        rp, ci = gg.single(loop)
        out = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=100)
        assert out["x"][0] == 1.0 and out["l1"] == 0.0


def test_first_update_on_tiny_by_hand(built_oracle):
    """One update on the 6-vertex graph in exact rational arithmetic.
    Out-degrees 2,2,1,1,0,3; vertex 4 dangling; x0 = 1/6 everywhere."""
    from fractions import Fraction as F
    rp, ci = tiny6()
    d = F(17, 20)
    x0 = F(1, 6)
    Dm = x0                                   # only vertex 4 is dangling
    sums = {0: x0 / 1 + x0 / 3,               # from 2 (outdeg 1) and 5 (outdeg 3)
            1: x0 / 2,                        # from 0
            2: x0 / 2 + x0 / 2,               # from 0 and 1
            3: x0 / 2 + x0 / 3,               # from 1 and 5
            4: x0 / 1 + x0 / 3,               # from 3 and 5
            5: F(0)}
    expect = [float((1 - d) / 6 + d * (sums[v] + Dm / 6)) for v in range(6)]
    out = oracle.pagerank(rp, ci, 0.85, tol=0.0, max_iter=1)
    np.testing.assert_allclose(out["x"], expect, rtol=1e-15)


def test_day40_case_sizes():
    for name, n, nnz in read_golden("day40_cases.txt"):
        rp, ci = day40_case(name)
        assert len(rp) - 1 == int(n) and len(ci) == int(nnz), name


# ----------------------------------------------- a planted mistake is caught --

MUTATIONS = [
    # D/n moved outside the d*(...) bracket
    ("x_next[v] = (1.0 - d) / nd + d * (s + D / nd);",
     "x_next[v] = (1.0 - d) / nd + d * s + D / nd;"),
    # dangling term dropped
    ("x_next[v] = (1.0 - d) / nd + d * (s + D / nd);",
     "x_next[v] = (1.0 - d) / nd + d * s;"),
    # divides by the in-degree of v instead of the out-degree of u
    ("s += x[u] / (double)outdeg[u];",
     "s += x[u] / (double)(in_ptr[v + 1] - in_ptr[v]);"),
    # pushes along out-edges instead of pulling along in-edges (transposed operand)
    ("int32_t u = in_col[j];", "int32_t u = (j < m) ? col_idx[j] : 0;"),
]


def _build_mutant(src_text, tmpdir, i):
    path = os.path.join(tmpdir, f"mut{i}.c")
    with open(path, "w") as f:
        f.write(src_text)
    so = os.path.join(tmpdir, f"mut{i}.so")
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", so, path, "-lm"], check=True)
    lib = ctypes.CDLL(so)
    i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
    lib.oracle_pagerank.argtypes = [i64, i64, vp, vp, dbl, dbl, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.oracle_pagerank.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("i", range(len(MUTATIONS)))
def test_planted_mistakes_fail_the_pins(built_oracle, i):
    """Plants each mistake in a copy of the oracle (CPU only) and checks that
    the dense brute-force pin rejects it."""
    with open(os.path.join(os.path.dirname(oracle.__file__), "pagerank_oracle.c")) as f:
        text = f.read()
    old, new = MUTATIONS[i]
    assert old in text
    with tempfile.TemporaryDirectory() as td:
        lib = _build_mutant(text.replace(old, new), td, i)
        rp, ci = gg.random_digraph(30, 0.15, 0.2, seed=31)
        rp = np.ascontiguousarray(rp, dtype=np.int64)
        ci = np.ascontiguousarray(ci, dtype=np.int32)
        n = 30
        x = np.empty(n)
        it = ctypes.c_int32(0)
        l1 = ctypes.c_double(0)
        p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        lib.oracle_pagerank(n, len(ci), p(rp), p(ci), 0.85, 0.0, 5, 0, None, p(x),
                            ctypes.byref(it), ctypes.byref(l1), None, None, None)
        G, _ = dense_google(rp, ci, D)
        y = np.full(n, 1.0 / n)
        for _ in range(5):
            y = G @ y
        assert not np.allclose(x, y, rtol=1e-9, atol=1e-12)
