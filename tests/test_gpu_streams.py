"""Handles on their own streams, from their own host threads.

Separate handles share nothing but the library's device memory pool, and the
update kernel never waits on another CTA, so two runs may overlap on the GPU.
Each run's result must equal, bit for bit, the same run done alone on the
default stream (runs are deterministic). One handle used from two streams in
sequence (ordered by the caller) must also give the same ranks.
"""
import threading

import numpy as np
import pytest

import graphgen as gg

torch = pytest.importorskip("torch")
import pagerank_power_iteration_gb300 as prg  # noqa: E402

pytestmark = pytest.mark.gpu
D = 0.85


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from pagerank_power_iteration_gb300 import build
    build.build()


def alone(rp, ci, dtype):
    with prg.Graph(rp, ci) as g:
        x, it, l1, _ = g.run(D, 1e-6, 200, dtype=dtype)
        ip, ic = g.in_csr()
    return x.cpu().numpy(), it, l1, ip, ic


def test_two_handles_on_two_streams_from_two_threads():
    graphs = [gg.workload("rmat18"), gg.citation(n=30000, seed=1)]
    dtypes = [torch.float32, torch.float64]
    ref = [alone(rp, ci, dt) for (rp, ci), dt in zip(graphs, dtypes)]
    results = [None, None]
    errors = []

    def work(k):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                rp, ci = graphs[k]
                rpd = torch.from_numpy(rp).cuda()
                cid = torch.from_numpy(ci).cuda()
                for _ in range(3):
                    with prg.Graph(rpd, cid, stream=st.cuda_stream) as g:
                        x, it, l1, _ = g.run(D, 1e-6, 200, dtype=dtypes[k], stream=st.cuda_stream)
                        ip, ic = g.in_csr(stream=st.cuda_stream)
                    st.synchronize()
                results[k] = (x.cpu().numpy(), it, l1, ip, ic)
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for got, exp in zip(results, ref):
        assert got[1] == exp[1]
        assert got[2] == exp[2]
        assert np.array_equal(got[0], exp[0])
        assert np.array_equal(got[3], exp[3]) and np.array_equal(got[4], exp[4])


def test_one_handle_on_two_streams_in_sequence():
    rp, ci = gg.rmat(14, seed=6)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with prg.Graph(rp, ci, stream=s1.cuda_stream) as g:
        x1, it1, _, _ = g.run(D, 1e-6, 200, stream=s1.cuda_stream)
        s1.synchronize()
        x2, it2, _, _ = g.run(D, 1e-6, 200, stream=s2.cuda_stream)
        s2.synchronize()
        x3, it3, _, _ = g.run(D, 1e-6, 200)
    assert it1 == it2 == it3
    assert torch.equal(x1, x2) and torch.equal(x1, x3)
