"""The random-gather rate measurement (the denominator of the update's gather
roofline): it runs, gives a finite positive rate in a plausible range for both
element types and for every request path (the warps' loads, the TMA's
tile::gather4 copies, both at once), and the update's own rate of gathers
from L2 on a graph whose state does not fit in shared memory stays below what
the measurement reports for a state of the same size (the update gathers and
does more besides)."""
import math

import pytest

import graphgen as gg

torch = pytest.importorskip("torch")
import pagerank_power_iteration_gb300 as prg  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from pagerank_power_iteration_gb300 import build
    build.build()


@pytest.mark.parametrize("path", [prg.PR_GATHER_LOAD, prg.PR_GATHER_TMA, prg.PR_GATHER_BOTH])
@pytest.mark.parametrize("dtype", [prg.PR_F32, prg.PR_F64])
@pytest.mark.parametrize("n", [1, 1000, 1 << 22])
def test_rate_is_finite_and_plausible(n, dtype, path):
    rate = prg.pr_measure_gather_rate(n, dtype, 1 << 24, None, path)
    assert math.isfinite(rate)
    # a random gather costs at least one cycle of an SM's L1: no GPU reaches
    # 10^13 per second, and anything below 10^9 would mean the kernel did not run
    assert 1e9 < rate < 1e13


@pytest.mark.parametrize("path", [prg.PR_GATHER_LOAD, prg.PR_GATHER_TMA, prg.PR_GATHER_BOTH])
def test_odd_gather_count(path):
    assert prg.pr_measure_gather_rate(4097, prg.PR_F32, 1001, None, path) > 0


def test_update_gathers_stay_below_the_measured_rate():
    rp, ci = gg.workload("rmat18")
    n, m = len(rp) - 1, len(ci)
    with prg.Graph(rp, ci) as g:
        g.run(0.85, 0.0, 20, dtype=torch.float32)
        stats = g.last_run()
        info = g.info()
    per_update = stats["loop_ms"] * 1e-3 / stats["iterations"]
    l2 = m - info["edges_hot_f32"]
    assert l2 > 0
    achieved = l2 / per_update
    rate = prg.pr_measure_gather_rate(n, prg.PR_F32, 1 << 27)
    assert achieved < 1.05 * rate, (achieved, rate)
