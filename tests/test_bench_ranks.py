"""The bench's multi-rank logic on CPU (gloo, world size 2): timings are reduced to the slowest
rank, the whole-job value counts every rank's batch, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 3.0 - rank]           # rank 1 is slower in the first entry, faster in the second
        q.put((rank, bench.max_over_ranks(mine, world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [11.0, 3.0]


def test_single_rank_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]


def test_job_value_counts_every_replica():
    one = bench.job_gbs(1, 62e6, 60e-6)
    assert abs(one - 1033.33) < 0.01
    assert abs(bench.job_gbs(4, 62e6, 60e-6) - 4 * one) < 1e-9


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 0, "gpus": 2})()
    assert bench.bench_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_keeps_the_contract(monkeypatch, capsys):
    # rank 0 prints one JSON line with the keys the driver reads, on the main workload's metric
    import json
    monkeypatch.setenv("RANK", "0")
    args = type("A", (), {"steps": 1, "warmup": 0, "gpus": 1})()
    assert bench.bench_reference(args) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["config"]["workload"] == bench.WORKLOAD and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
