"""The multi-rank path of bench.py on CPU (gloo, world size 2): every rank
runs its own replica of the step; the job's time is the slowest rank's and
its throughput counts the units of all ranks.  No data-path collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        assert bench.env_rank() == (rank, rank, world)
        # rank r's replica took 1+r ms for the step and 0.5+2r ms for its kernel
        got = bench.max_over_ranks([1.0 + rank, 0.5 + 2 * rank], "cpu")
        rate = bench.whole_job_rate(1e9, world, got[0])
        out[rank] = (got, rate)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_world_2():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        got, rate = res[rank]
        assert got == [2.0, 2.5]
        assert rate == pytest.approx(1e9 * 2 / 2e-3)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.whole_job_rate(10.0, 1, 1.0) == pytest.approx(1e4)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload = "tiny_T12_hq4_hkv2_d64"
        steps = 1
        warmup = 0
    bench.run_reference(A())
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_line(monkeypatch, capsys):
    import json

    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class A:
        workload = "tiny_T12_hq4_hkv2_d64"
        steps = 2
        warmup = 1
    bench.run_reference(A())
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["metric"] == bench.METRIC
