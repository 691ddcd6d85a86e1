"""Host-side pieces of bench.py (no GPU): the byte model against the Day 40
page's printed figures, the CPU sample, and the N>1 aggregation over two gloo
ranks on the CPU."""
import math
import os
import socket

import numpy as np
import pytest

import bench
import graphgen as gg
from conftest import read_golden


def golden_measurements():
    return {k: float(v) for k, v in read_golden("day40_measurements.txt")}


def test_byte_model_reproduces_day40_figures():
    g = golden_measurements()
    b = bench.day40_bytes(int(g["nodes"]), int(g["edges"]))
    assert b["hand"] == int(g["bytes_hand"])
    assert b["library"] == int(g["bytes_library"])
    assert b["library"] / b["hand"] == pytest.approx(1.80, abs=0.005)


def test_sum_tolerance_rule():
    g = golden_measurements()
    flt_eps = float(np.finfo(np.float32).eps)
    assert 4 * flt_eps * math.sqrt(g["nodes"]) == pytest.approx(g["sum_tolerance"], rel=1e-3)


def test_spmv_byte_model():
    bm = bench.bytes_model(16, 100)
    assert bm["b_spmv"] == 4 * 17 + 8 * 100 + 4 * 16
    assert bm["b_floor"] == 4 * 17 + 4 * 100 + 8 * 16


def test_prefix_sample_is_a_prefix_of_the_edge_stream():
    rp, ci = gg.rmat(12, seed=3)
    srp, sci = bench.prefix_sample(rp, ci, 20000)
    assert len(srp) == len(rp) and srp[-1] == len(sci) <= 20000
    assert np.array_equal(sci, ci[: len(sci)])
    assert np.all(np.diff(srp) >= 0)
    full = bench.prefix_sample(rp, ci, 10 ** 9)
    assert full[1] is ci


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--workload", "citation30k"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_line(monkeypatch, capsys):
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--impl", "reference", "--workload", "citation30k", "--steps", "2", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "GTEPS" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, edges = bench.aggregate(dist, "cpu", 10.0 + 5.0 * rank, 1000.0 * (rank + 1))
        q.put((rank, ms, edges))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, edges in got:
        assert ms == 15.0 and edges == 3000.0


def test_aggregate_without_process_group():
    assert bench.aggregate(None, "cpu", 12.5, 77.0) == (12.5, 77.0)


def test_code_digest_ignores_comments_but_not_code():
    import bench
    a = "int f(int x) {\n    return x + 1;   // add one\n}\n"
    b = "/* header */\nint f(int x) {\n\n    return x + 1;\n}\n"
    c = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench.code_digest(a) == bench.code_digest(b)
    assert bench.code_digest(a) != bench.code_digest(c)
