import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


def read_golden(name):
    """Lines of a golden fixture with comments and blank lines removed."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


def simple_dataset_11():
    """The 11-vertex sample graph from the @antv/page-rank notebook, as CSR."""
    import graphgen as gg
    pairs = read_golden("simple_dataset_11.txt")
    src = [ord(a) - ord("A") for a, _ in pairs]
    dst = [ord(b) - ord("A") for _, b in pairs]
    return gg.from_edges(11, src, dst)


def tiny6():
    """A 6-vertex, 9-edge graph with one dangling vertex (4), sized like the
    Day 40 'tiny' case."""
    import graphgen as gg
    edges = [(0, 1), (0, 2), (1, 2), (1, 3), (2, 0), (3, 4), (5, 3), (5, 4), (5, 0)]
    return gg.from_edges(6, [e[0] for e in edges], [e[1] for e in edges])


def dangling4096():
    """Day 40 'dangling' case sizes: the (1, 2) circulant on 4096 vertices with
    400 seeded vertices stripped of their out-edges (8192 - 800 = 7392 edges)."""
    import graphgen as gg
    n = 4096
    rng = np.random.default_rng(40)
    dead = np.zeros(n, dtype=bool)
    dead[rng.choice(n, size=400, replace=False)] = True
    u = np.arange(n)
    src = np.concatenate([u, u])
    dst = np.concatenate([(u + 1) % n, (u + 2) % n])
    keep = ~dead[src]
    return gg.from_edges(n, src[keep], dst[keep])


def day40_case(name):
    import graphgen as gg
    if name == "tiny":
        return tiny6()
    if name == "single":
        return gg.single()
    if name == "nodangling":
        return gg.circulant(4096, (1, 2))
    if name == "dangling":
        return dangling4096()
    if name == "star":
        return gg.star_in(10000)
    if name == "chain":
        return gg.chain(8192)
    raise KeyError(name)


@pytest.fixture(scope="session")
def built_oracle():
    import oracle
    oracle.build()
    return oracle
