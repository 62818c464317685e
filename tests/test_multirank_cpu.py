"""The N-GPU bench path on CPU: N independent replicas over a gloo process
group (world size 2), whole-job timing = the slowest rank's time and the
tokens of all ranks; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [10.0, 12.5][rank]
    toks = [100.0, 150.0][rank]
    dist.barrier()
    out = bench.reduce_over_ranks(dist, ms, toks, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out))


def test_replica_timing_reduces_max_time_and_total_tokens():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == (12.5, 250.0) and res[1] == (12.5, 250.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    class Args:
        config, ctx, skip, gamma, steps, warmup = "tiny", 64, 0.5, 3, 1, 1

    monkeypatch.setenv("RANK", "1")
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
