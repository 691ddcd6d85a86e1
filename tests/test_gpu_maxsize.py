"""The largest graph pr_graph_create accepts for n = 2^24: m = max_edges(n)
(about 2.1e9 edges, m + 3n + PR_LAYOUT_SLACK = 2^31 - 1), so every int32
offset of the transpose and of the padded work layout is at its limit.

The graph is generated on the device (row_ptr[u] = floor(u m / n), targets
uniform from a seeded generator; every vertex has out-degree 124 or 125, no
dangling vertex). At this size the oracle cannot run, so the checks are the
ones that hold at any size, computed on the device in int64/fp64:
- in_ptr[n] = m and the in-degrees equal a histogram of col_idx;
- sampled in-rows equal the sources of the edges into that vertex, ascending;
- one update from the uniform start equals the update formula on the sampled
  rows, and the ranks sum to 1; a converged run also sums to 1.
About 60 GB of device memory at peak.
"""
import pytest

torch = pytest.importorskip("torch")
import pagerank_power_iteration_gb300 as prg  # noqa: E402
from gpu_util import F32  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
D = 0.85


@pytest.fixture(scope="module")
def graph():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from pagerank_power_iteration_gb300 import build
    build.build()
    n = 1 << 24
    m = prg.max_edges(n)
    assert m + 3 * n + prg.PR_LAYOUT_SLACK == (1 << 31) - 1
    dev = torch.device("cuda:0")
    rp = torch.arange(n + 1, dtype=torch.int64, device=dev) * m // n
    gen = torch.Generator(device=dev).manual_seed(12)
    ci = torch.randint(0, n, (m,), dtype=torch.int32, device=dev, generator=gen)
    g = prg.Graph(rp, ci)
    yield n, m, rp, ci, g
    g.close()
    del ci, rp
    torch.cuda.empty_cache()


def sources_into(rp, ci, v):
    """Sources of the edges into v, in out-CSR order (ascending)."""
    j = (ci == v).nonzero().flatten()
    return torch.searchsorted(rp, j, right=True) - 1


def test_transpose_at_the_int32_limit(graph):
    n, m, rp, ci, g = graph
    info = g.info()
    assert info["n"] == n and info["m"] == m and info["n_dangling"] == 0
    in_ptr = torch.empty(n + 1, dtype=torch.int32, device="cuda")
    in_col = torch.empty(m, dtype=torch.int32, device="cuda")
    prg.pr_get_in_csr(g.handle, in_ptr.data_ptr(), in_col.data_ptr(), None)
    torch.cuda.synchronize()
    assert int(in_ptr[0]) == 0 and int(in_ptr[-1]) == m
    indeg = torch.diff(in_ptr.long())
    assert torch.equal(indeg, torch.bincount(ci, minlength=n))
    for v in [0, 1, n // 2, n - 1, int(torch.argmax(indeg)), 12345]:
        row = in_col[in_ptr[v]:in_ptr[v + 1]].long()
        assert torch.equal(row, sources_into(rp, ci, v)), v


def test_one_update_and_a_converged_run_at_the_int32_limit(graph):
    n, m, rp, ci, g = graph
    x, it, _, _ = g.run(D, 0.0, 1)
    assert it == 1
    outdeg = torch.diff(rp).double()
    for v in [0, 7, n // 3, n - 1, 424242]:
        src = sources_into(rp, ci, v)
        y = torch.sum(1.0 / (n * outdeg[src])).item()
        want = (1.0 - D) / n + D * y          # no dangling vertex: D = 0
        got = float(x[v])
        assert abs(got - want) <= F32["rel"] * abs(want) + F32["abs"], (v, got, want)
    assert abs(float(x.double().sum()) - 1.0) <= F32["sum"]
    x, it, l1, conv = g.run(D, 1e-6, 200)
    assert conv and l1 < 1e-6 and 1 < it < 200
    assert abs(float(x.double().sum()) - 1.0) <= F32["sum"]
