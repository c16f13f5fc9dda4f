"""Host logic of bench.py's multi-GPU mode (replicas only), on CPU with gloo.

Each rank times its own replica; the job's time is the slowest rank's (a
MAX all-reduce) and the whole-job rate counts every rank's steps.  Under
torchrun the reference arm runs on rank 0 alone; the other ranks exit without
work or output.
"""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(dist, 10.0 + 5.0 * rank, "cpu")   # rank 1 is the slow one
    out.put((rank, ms, bench.whole_job_rate(world, 4, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_time_is_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    assert all(abs(r[2] - 2 * 4 / 0.015) < 1e-9 for r in res)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 12.5, "cpu") == 12.5
    assert bench.whole_job_rate(1, 10, 2000.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from long_context_speculative_gb300 import workloads as wl

    calls = []

    def fake_sample(w):
        calls.append(w.name)
        return 2.0, 4, "fake sample", 2.0

    monkeypatch.setattr(bench, "oracle_sample_time", fake_sample)
    args = type("A", (), {"gpus": 2, "steps": 2, "warmup": 1})()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(args, wl.LLAMA8B_120K)
    assert capsys.readouterr().out == "" and calls == []
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(args, wl.LLAMA8B_120K)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["value"] == pytest.approx(0.5)
    assert line["n_gpus"] == 2 and len(calls) == 2
