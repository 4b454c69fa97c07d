"""Multi-process (gloo, CPU) tests of bench.py's replica aggregation: the
slowest rank's timed region sets the time, the value counts every rank's
units, and the reference arm runs on rank 0 only."""
import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    region = [10.0, 25.0][rank]
    m = bench.max_over_ranks(region, world)
    rate = bench.whole_job_rate(1000, 4, world, m)
    q.put((rank, m, rate))
    dist.destroy_process_group()


def test_two_rank_max_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29613
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, rate in got:
        assert m == 25.0
        assert rate == pytest.approx(2 * 1000 * 4 / 0.025)


def test_reference_arm_non_zero_rank_exits_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        gpus, steps, warmup = 2, 3, 1
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(10, 2, 1, 1000.0) == pytest.approx(20.0)

def test_reference_arm_rank0_line(monkeypatch, capsys):
    """The oracle arm on the host cores: one JSON line with the contract's keys,
    the whole decode batch per step and the GPU arm's config object."""
    sys.path.insert(0, ROOT)
    import json
    import bench
    from deterministic_paged_kv_gb300 import workloads
    monkeypatch.setenv("RANK", "0")

    class A:
        gpus, steps, warmup = 1, 1, 0
    assert bench.run_reference(A()) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = workloads.decode_throughput()
    step_bytes = bench.decode_alg_bytes(w)
    assert line["impl"] == "reference" and line["metric"] == "paged decode HBM GB/s"
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True and line["steps"] == 1
    assert line["config"] == bench.decode_step_config(w, step_bytes, 1)
    assert line["value"] > 0 and line["value"] == pytest.approx(step_bytes / (line["ms_per_step"] * 1e-3) / 1e9)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
