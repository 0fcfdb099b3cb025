"""Host logic of the multi-rank benchmark on CPU ranks (gloo, world size 2):
the slowest rank's time is what every rank reports, each rank draws its own
batch, and the reference arm runs on rank 0 only."""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from mxfp4_activation_quant_gb300 import synth

        t = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
        w = bench.rank_workload(synth.WORKLOADS["prefill"], rank)
        x = synth.make_inputs(w, M=2)["x"]
        dist.barrier()
        q.put((rank, t, w.seed, x.float().sum().item()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_draw_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, q), nprocs=2, start_method="spawn", join=True)
    got = sorted(q.get() for _ in range(2))
    assert [g[1] for g in got] == [15.0, 15.0]
    assert got[0][2] != got[1][2] and got[0][3] != got[1][3]


def test_reference_arm_is_silent_on_other_ranks(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 3, "gpus": 2})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""
