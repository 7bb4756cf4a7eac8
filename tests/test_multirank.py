"""Multi-rank benchmark logic on CPU (gloo, world size 2): each rank runs its
own GEMM (weak scaling, no exchange on the data path); the job's step time is
the slowest rank's and the reported value aggregates every rank's work."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 1.0 + rank * 0.5                      # rank 1 is slower
    got = bench.max_over_ranks(ms, dist, torch, "cpu")
    out.put((rank, got, bench.aggregate_tflops(world, 2.0e12, got)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value_gloo():
    import socket

    import torch.multiprocessing as mp
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [1.5, 1.5]
    # 2 ranks x 2e12 flop in 1.5 ms
    assert abs(res[0][2] - 2 * 2.0e12 / 1.5e-3 / 1e12) < 1e-9


def test_reference_arm_prints_only_on_rank0(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), dict(workload="bs_tiny_256x512x512", seed=0, steps=1, warmup=1, gpus=2,
                              cpu_seconds=1.0, ref_seconds=5.0))()
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_rank0(capsys, monkeypatch):
    import json
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    args = type("A", (), dict(workload="bs_tiny_256x512x512", seed=0, steps=2, warmup=1, gpus=1,
                              cpu_seconds=1.0, ref_seconds=5.0))()
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    # nothing extrapolated: the per-step time is the measured one, for the rows the line names
    assert line["extrapolated"] is False and line["ms_per_step"] > 0 and 1 <= line["rows_per_step"] <= 256
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
