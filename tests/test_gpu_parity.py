"""Parity of the CUDA path (through the C ABI) against the oracle.

The transpose must be bit-exact. Ranks are compared at the same number of
updates (the oracle is rerun with that fixed count); converged iteration
counts must agree within one update.
"""
import numpy as np
import pytest

import graphgen as gg
import oracle
from conftest import day40_case
from gpu_util import F32, F64, assert_ranks_close

torch = pytest.importorskip("torch")
import pagerank_power_iteration_gb300 as prg  # noqa: E402

pytestmark = pytest.mark.gpu
D = 0.85


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from pagerank_power_iteration_gb300 import build
    build.build()
    oracle.build()


def graph_with_in_degrees(degs, n, seed):
    """A graph on n vertices whose first len(degs) vertices (in a shuffled order)
    have the given in-degrees, from distinct random sources; the other vertices
    have no in-edges. Out-degrees follow from the draw (some sources dangle)."""
    rng = np.random.default_rng(seed)
    rows = rng.permutation(n)[: len(degs)]
    src, dst = [], []
    for v, k in zip(rows, degs):
        src.append(rng.choice(n, size=k, replace=False))
        dst.append(np.full(k, v))
    return gg.from_edges(n, np.concatenate(src), np.concatenate(dst))


def layout_degrees():
    """In-degrees that cover the work layout's edges: every thread-class length
    1..32 (so 32-row blocks mix padded lengths and the split between long and
    short blocks falls inside a block), warp-class rows at the 4-edge padding
    and 128-edge step boundaries up to 1024, hub rows around the 256-edge
    chunks, and a row count that is not a multiple of 32."""
    degs = list(range(1, 33)) * 37
    degs += [33, 34, 35, 36, 64, 127, 128, 129, 255, 256, 511, 512, 513, 1000, 1023, 1024] * 3
    degs += [1025, 1536, 2048, 2049, 5000]
    return degs


def graph(name):
    if name == "layout":
        return graph_with_in_degrees(layout_degrees(), 9011, seed=7)
    if name == "t_short_only":   # thread-class rows of one or two int4s only
        return graph_with_in_degrees([1 + i % 8 for i in range(999)], 4001, seed=8)
    if name == "t_long_only":    # thread-class rows of three to eight int4s only
        return graph_with_in_degrees([9 + i % 24 for i in range(1001)], 4003, seed=9)
    if name in ("tiny", "single", "nodangling", "dangling", "star", "chain"):
        return day40_case(name)
    if name == "star_out":
        return gg.star_out(10000)
    if name == "no_edges":
        return gg.from_edges(5, [], [])
    if name == "all_dangling_but_one":
        return gg.from_edges(300, [7, 7], [3, 250])
    if name == "selfloops1":
        return gg.from_edges(1, [0, 0, 0], [0, 0, 0])
    if name == "dups_loops":
        return gg.random_sparse(3000, 40000, seed=11, dangling_frac=0.3)
    if name == "hub70k":
        return gg.star_in(70000)
    if name == "n257":
        return gg.random_sparse(257, 3000, seed=3)
    if name == "n65537":
        return gg.random_sparse(65537, 300000, seed=4, dangling_frac=0.1)
    if name == "citation30k":
        return gg.workload("citation30k")
    if name == "rmat14":
        return gg.rmat(14, seed=6)
    if name == "rmat18":
        return gg.workload("rmat18")
    if name == "er16":
        return gg.erdos_renyi(1 << 16, 16, 0.1, seed=5)
    raise KeyError(name)


SMALL = ["tiny", "single", "nodangling", "dangling", "star", "chain", "star_out", "no_edges",
         "all_dangling_but_one", "selfloops1", "dups_loops", "hub70k", "n257", "n65537",
         "citation30k", "rmat14", "er16", "layout", "t_short_only", "t_long_only"]


@pytest.mark.parametrize("name", SMALL + ["rmat18"])
def test_transpose_bit_exact(name):
    rp, ci = graph(name)
    with prg.Graph(rp, ci) as g:
        ip, ic = g.in_csr()
        info = g.info()
    oip, oic = oracle.transpose(rp, ci)
    assert np.array_equal(ip.astype(np.int64), oip)
    assert np.array_equal(ic, oic)
    indeg = np.diff(oip)
    assert info["rows_zero"] == int((indeg == 0).sum())
    assert info["rows_thread"] == int(((indeg >= 1) & (indeg <= 32)).sum())
    assert info["rows_warp"] == int(((indeg > 32) & (indeg <= 1024)).sum())
    assert info["rows_cta"] == int((indeg > 1024).sum())
    assert info["edges_cta"] == int(indeg[indeg > 1024].sum())
    assert info["n_dangling"] == int((np.diff(rp) == 0).sum())


def test_four_radix_passes():
    """n > 2^24 needs a fourth 8-bit pass: the first writes (destination,
    source) pairs, two middle passes (digits at bits 8 and 16) read and write
    them, and the last (bits 24-31) writes the sources. Sparse, so that the
    oracle's n-bin counting sort and updates stay quick."""
    n = (1 << 24) + (1 << 20)
    rp, ci = gg.random_sparse(n, 4_000_000, seed=13, dangling_frac=0.5)
    assert (ci >= 1 << 24).sum() > 10000   # the top digit is not always 0
    with prg.Graph(rp, ci) as g:
        ip, ic = g.in_csr()
    oip, oic = oracle.transpose(rp, ci)
    assert np.array_equal(ip.astype(np.int64), oip)
    assert np.array_equal(ic, oic)
    _parity(rp, ci, "f32")


def work_order(rp, ci):
    """The documented class-major work order, derived independently on the host:
    rows with in-degree > 1024, then 33..1024, then 1..32, then 0; inside the
    first two classes by half-octave bucket of the out-degree, largest first;
    thread-class rows by padded length in int4s (longest first), then by a coarse
    out-degree bucket; ties by vertex id."""
    n = len(rp) - 1
    indeg = np.bincount(ci, minlength=n).astype(np.int64)
    outdeg = np.diff(rp).astype(np.int64)
    cls = np.select([indeg > 1024, indeg > 32, indeg > 0], [0, 1, 2], 3)
    x = outdeg + 1
    b = np.floor(np.log2(x)).astype(np.int64)
    half = np.where(b > 0, (x >> np.maximum(b - 1, 0)) & 1, 0)
    ob = np.minimum(63, 2 * b + half)
    sub = np.where(cls == 2, (8 - ((indeg + 3) >> 2)) * 8 + (7 - np.minimum(7, ob >> 2)), 63 - ob)
    return np.argsort(cls * 64 + sub, kind="stable")


@pytest.mark.parametrize("name", ["layout", "rmat18", "citation30k"])
def test_hot_source_edge_counts(name):
    """edges_hot_* counts the in-edges whose source is among the first 40,960
    (fp32) or 20,480 (fp64) vertices of the work order: every out-edge of such a
    vertex, so the count is the sum of their out-degrees."""
    rp, ci = graph(name)
    with prg.Graph(rp, ci) as g:
        info = g.info()
    outdeg = np.diff(rp)
    order = work_order(rp, ci)
    assert info["edges_hot_f32"] == int(outdeg[order[:40960]].sum())
    assert info["edges_hot_f64"] == int(outdeg[order[:20480]].sum())
    assert 0 <= info["edges_hot_f64"] <= info["edges_hot_f32"] <= info["m"]


def _parity(rp, ci, dtype, tol=1e-6, max_iter=200, check_iters=True):
    tt = {"f32": torch.float32, "f64": torch.float64}[dtype]
    tolset = F32 if dtype == "f32" else F64
    with prg.Graph(rp, ci) as g:
        x, it, l1, conv = g.run(D, tol, max_iter, dtype=tt)
        x = x.cpu().numpy()
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=it)
    assert_ranks_close(x, ref["x"], tolset, f"{dtype} after {it} updates")
    assert abs(x.sum() - 1.0) <= tolset["sum"]
    # L1 is a sum of |x' - x| over values rounded to the rank precision: each
    # term can be off by about ulp(x'[v]) + ulp(x[v]) <= 2 * eps * x[v], so
    # the total by up to 2 * 2 * eps * sum(x) = 4 * eps (eps = 2^-23 in fp32).
    l1_floor = 4 * 2.0 ** -23 if dtype == "f32" else 1e-12
    assert abs(l1 - ref["l1"]) <= max(0.02 * ref["l1"], l1_floor)
    if check_iters and tol > 0:
        refc = oracle.pagerank(rp, ci, D, tol=tol, max_iter=max_iter)
        assert abs(refc["iters"] - it) <= 1, (refc["iters"], it)
        assert conv == (refc["status"] == oracle.OK) or abs(refc["iters"] - it) == 1
    return it


@pytest.mark.parametrize("name", SMALL + ["rmat18"])
def test_converged_ranks_f32(name):
    rp, ci = graph(name)
    _parity(rp, ci, "f32")


@pytest.mark.parametrize("name", ["tiny", "dangling", "star", "chain", "dups_loops", "hub70k", "layout",
                                  "citation30k", "rmat14", "er16", "layout", "t_short_only", "t_long_only"])
def test_converged_ranks_f64(name):
    rp, ci = graph(name)
    _parity(rp, ci, "f64", tol=1e-10, max_iter=400)


@pytest.mark.parametrize("name", ["dangling", "citation30k", "rmat14", "layout"])
@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_fixed_iterations(name, dtype):
    """tol <= 0 runs exactly max_iter updates (the timed fixed-50 mode)."""
    rp, ci = graph(name)
    tt = {"f32": torch.float32, "f64": torch.float64}[dtype]
    # odd and even counts: the graph's loop runs two update launches per
    # trip, and a trip that ends on its first update must not run the second
    for k in (1, 2, 3, 7, 50):
        with prg.Graph(rp, ci) as g:
            x, it, l1, conv = g.run(D, 0.0, k, dtype=tt)
            stats = g.last_run()
        assert it == k and conv and stats["iterations"] == k
        assert stats["launches"] == (k + 1) // 2 * 2 + 2   # init, the loop's launches, output
        ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=k)
        assert_ranks_close(x.cpu().numpy(), ref["x"], F32 if dtype == "f32" else F64, f"k={k}")


def test_closed_forms_on_device():
    """Cycle: 1/n after one update; star (leaves -> centre): the closed form."""
    rp, ci = gg.cycle(100000)
    with prg.Graph(rp, ci) as g:
        x, it, l1, conv = g.run(D, 1e-6, 200)
    assert it == 1 and conv
    assert np.allclose(x.cpu().numpy(), 1.0 / 100000, rtol=1e-6, atol=0)
    k = 10000
    rp, ci = gg.star_in(k)
    with prg.Graph(rp, ci) as g:
        x, it, l1, conv = g.run(D, 1e-9, 500, dtype=torch.float64)
    xc = (1 + k * D) / (1 + k + k * D)
    assert abs(x[0].item() - xc) < 1e-9


@pytest.mark.parametrize("d", [0.0, 0.5, 1.0])
def test_damping_extremes(d):
    rp, ci = graph("dangling")
    with prg.Graph(rp, ci) as g:
        x, it, l1, conv = g.run(d, 0.0, 20, dtype=torch.float64)
    ref = oracle.pagerank(rp, ci, d, tol=0.0, max_iter=20)
    assert_ranks_close(x.cpu().numpy(), ref["x"], F64, f"d={d}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_warm_start(dtype):
    rp, ci = graph("citation30k")
    tt = {"f32": torch.float32, "f64": torch.float64}[dtype]
    rng = np.random.default_rng(3)
    x0 = rng.random(len(rp) - 1)
    x0 /= x0.sum()
    with prg.Graph(rp, ci) as g:
        xi = torch.tensor(x0, dtype=tt, device="cuda")
        x, it, l1, conv = g.run(D, 0.0, 7, dtype=tt, x_init=xi)
        xh, _, _, _ = g.run(D, 0.0, 7, dtype=tt, x_init=x0.astype(np.float32 if dtype == "f32" else np.float64))
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=7, x_init=x0)
    tol = F32 if dtype == "f32" else F64
    assert_ranks_close(x.cpu().numpy(), ref["x"], tol, "device x_init")
    assert_ranks_close(xh.cpu().numpy(), ref["x"], tol, "host x_init")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_isolated_vertices(dtype):
    """Vertices with neither in- nor out-edges are combined row by row in the
    first update only; later updates count them as n_iso equal terms and the
    output gives them the last constant term. Half the vertices here are
    isolated; a warm start gives them arbitrary first values, so the first
    update's L1 and dangling terms differ per vertex. Every count of updates
    must match the oracle, and each isolated rank must be the constant term
    (1-d)/n + d D/n of the last update."""
    n = 6001
    rng = np.random.default_rng(21)
    live = rng.permutation(n)[: n // 2]
    src = rng.choice(live, size=20000)
    dst = rng.choice(live, size=20000)
    rp, ci = gg.from_edges(n, src, dst)
    outdeg, indeg = np.diff(rp), np.bincount(ci, minlength=n)
    iso = (outdeg == 0) & (indeg == 0)
    assert iso.sum() >= n // 2
    tt = {"f32": torch.float32, "f64": torch.float64}[dtype]
    tolset = F32 if dtype == "f32" else F64
    x0 = rng.random(n)
    x0 /= x0.sum()
    with prg.Graph(rp, ci) as g:
        for k in (1, 2, 3, 10):
            for start in (None, x0):
                xi = None if start is None else torch.tensor(start, dtype=tt, device="cuda")
                x, it, l1, _ = g.run(D, 0.0, k, dtype=tt, x_init=xi)
                x = x.cpu().numpy()
                ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=k,
                                      **({} if start is None else {"x_init": start}))
                assert_ranks_close(x, ref["x"], tolset, f"k={k} warm={start is not None}")
                l1_floor = 4 * 2.0 ** -23 if dtype == "f32" else 1e-12
                assert abs(l1 - ref["l1"]) <= max(0.02 * ref["l1"], l1_floor)
                assert np.all(x[iso] == x[iso][0])   # one constant term for all of them


def test_precisions_alternate_on_one_handle():
    """The fp32 state is made with the handle and the fp64 state on the first
    fp64 run; runs of the two precisions share the handle's scalars. Runs that
    alternate must each equal the same run on a fresh handle, bit for bit."""
    rp, ci = graph("rmat14")
    fresh = {}
    for tt in (torch.float32, torch.float64):
        with prg.Graph(rp, ci) as g:
            fresh[tt] = g.run(D, 1e-6, 200, dtype=tt)
    with prg.Graph(rp, ci) as g:
        for tt in (torch.float32, torch.float64, torch.float32, torch.float64, torch.float32):
            x, it, l1, conv = g.run(D, 1e-6, 200, dtype=tt)
            fx, fit, fl1, fconv = fresh[tt]
            assert it == fit and l1 == fl1 and conv == fconv
            assert torch.equal(x, fx)


def test_host_and_device_buffers_agree():
    rp, ci = graph("rmat14")
    with prg.Graph(rp, ci) as g:                      # host inputs
        xa, ita, _, _ = g.run(D, 1e-6, 200)
        host_out = np.empty(len(rp) - 1, dtype=np.float32)
        xb, itb, _, _ = g.run(D, 1e-6, 200, out=host_out)
    rpd = torch.from_numpy(rp).cuda()
    cid = torch.from_numpy(ci).cuda()
    with prg.Graph(rpd, cid) as g:                    # device inputs
        xc, itc, _, _ = g.run(D, 1e-6, 200)
    assert ita == itb == itc
    assert xb is host_out
    assert np.array_equal(xa.cpu().numpy(), host_out)
    assert np.array_equal(xa.cpu().numpy(), xc.cpu().numpy())


@pytest.mark.parametrize("name", ["rmat18", "citation30k", "hub70k", "layout"])
def test_runs_repeat_bit_for_bit(name):
    """Every sum is formed in a fixed order and L1 / D are exact fixed-point
    sums, so repeated runs (and a second handle) give identical bits."""
    rp, ci = graph(name)
    with prg.Graph(rp, ci) as g:
        a, ita, l1a, _ = g.run(D, 1e-6, 200)
        b, itb, l1b, _ = g.run(D, 1e-6, 200)
        c, itc, _, _ = g.run(D, 0.0, 5, dtype=torch.float64)
        c2, _, _, _ = g.run(D, 0.0, 5, dtype=torch.float64)
        e, ite, l1e, _ = g.run(D, 1e-6, 200)
        st = g.last_run()
    with prg.Graph(rp, ci) as g2:
        f, itf, l1f, _ = g2.run(D, 1e-6, 200)
    assert ita == itb == ite == itf and itc == 5
    assert l1a == l1b == l1e == l1f
    for other in (b, e, f):
        assert np.array_equal(a.cpu().numpy(), other.cpu().numpy())
    assert np.array_equal(c.cpu().numpy(), c2.cpu().numpy())
    assert st["iterations"] == ite and st["loop_ms"] > 0


def test_not_converged_status():
    rp, ci = graph("citation30k")
    with prg.Graph(rp, ci) as g:
        x, it, l1, conv = g.run(D, 1e-12, 3)
    assert it == 3 and not conv and l1 > 1e-12


def test_invalid_graphs_are_rejected():
    rp, ci = graph("tiny")
    bad = ci.copy(); bad[3] = 6
    with pytest.raises(prg.PageRankError) as e:
        prg.Graph(rp, bad)
    assert e.value.status == prg.PR_ERR_INVALID_GRAPH
    bad = ci.copy(); bad[0] = -2
    with pytest.raises(prg.PageRankError) as e:
        prg.Graph(torch.from_numpy(rp).cuda(), torch.from_numpy(bad).cuda())
    assert e.value.status == prg.PR_ERR_INVALID_GRAPH
    rbad = rp.copy(); rbad[2], rbad[3] = rbad[3], rbad[2]
    with pytest.raises(prg.PageRankError) as e:
        prg.Graph(rbad, ci)
    assert e.value.status == prg.PR_ERR_INVALID_GRAPH
    rbad = rp.copy(); rbad[-1] -= 1
    with pytest.raises(prg.PageRankError) as e:
        prg.Graph(rbad, ci)
    assert e.value.status == prg.PR_ERR_INVALID_GRAPH
    # the context is still usable afterwards
    with prg.Graph(rp, ci) as g:
        x, it, _, _ = g.run(D, 1e-6, 100)
    assert it > 1


def test_bad_row_ptr_while_host_col_idx_is_copied():
    """A host col_idx is copied on the library's second stream while the
    row_ptr-only steps run; a bad row_ptr stops the build there, with the copy
    (1.2 ms for RMAT-22's 261 MB) still in flight. The build must wait for it
    before its buffer goes back to the pool, and the next build from host
    arrays must equal one from device arrays."""
    rp, ci = gg.workload("rmat22")
    rbad = rp.copy()
    k = len(rbad) // 2
    rbad[k] = rbad[k + 1] + 1   # row_ptr decreases once; row_ptr[n] = m still
    for _ in range(3):
        with pytest.raises(prg.PageRankError) as e:
            prg.Graph(rbad, ci)
        assert e.value.status == prg.PR_ERR_INVALID_GRAPH
    with prg.Graph(rp, ci) as g:
        ip, ic = g.in_csr()
        x, it, _, _ = g.run(D, 1e-6, 200)
    with prg.Graph(torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda()) as g:
        ip2, ic2 = g.in_csr()
        x2, it2, _, _ = g.run(D, 1e-6, 200)
    assert np.array_equal(ip, ip2) and np.array_equal(ic, ic2)
    assert it == it2 and torch.equal(x, x2)


@pytest.mark.parametrize("thread_max,warp_max", [(1, 1), (8, 64), (32, 32), (16, 4096), (32, 8192)])
@pytest.mark.parametrize("name", ["layout", "hub70k", "dups_loops", "citation30k", "rmat14"])
def test_class_thresholds(name, thread_max, warp_max):
    """The class thresholds move rows between kernel paths only: the transpose
    is unchanged, the class sizes follow the thresholds, and the ranks agree
    with the oracle at the same number of updates."""
    rp, ci = graph(name)
    with prg.Graph(rp, ci, thread_max=thread_max, warp_max=warp_max) as g:
        ip, ic = g.in_csr()
        info = g.info()
        x, it, l1, conv = g.run(D, 1e-6, 200)
        x = x.cpu().numpy()
    oip, oic = oracle.transpose(rp, ci)
    assert np.array_equal(ip.astype(np.int64), oip) and np.array_equal(ic, oic)
    indeg = np.diff(oip)
    assert (info["thread_max"], info["warp_max"]) == (thread_max, warp_max)
    assert info["rows_thread"] == int(((indeg >= 1) & (indeg <= thread_max)).sum())
    assert info["rows_warp"] == int(((indeg > thread_max) & (indeg <= warp_max)).sum())
    assert info["rows_cta"] == int((indeg > warp_max).sum())
    assert info["edges_cta"] == int(indeg[indeg > warp_max].sum())
    assert info["edges_thread"] + info["edges_warp"] + info["edges_cta"] == len(ci)
    ref = oracle.pagerank(rp, ci, D, tol=0.0, max_iter=it)
    assert_ranks_close(x, ref["x"], F32, f"{name} thresholds {thread_max}/{warp_max}")
    refc = oracle.pagerank(rp, ci, D, tol=1e-6, max_iter=200)
    assert abs(refc["iters"] - it) <= 1


def test_build_stage_timing():
    rp, ci = graph("rmat18")
    with prg.Graph(rp, ci, stage_timing=True) as g:
        info = g.info()
    stages = info["build_stage_ms"]
    assert list(stages) == list(prg.BUILD_STAGES)
    assert all(v > 0.0 for v in stages.values()), stages
    total = sum(stages.values())
    # the stages tile the build from its first launch to its last
    assert info["build_ms"] > 0.0 and abs(total - info["build_ms"]) <= 0.02 * info["build_ms"] + 0.01
    with prg.Graph(rp, ci) as g:
        info = g.info()
    assert info["build_ms"] > 0.0 and all(v == 0.0 for v in info["build_stage_ms"].values())
