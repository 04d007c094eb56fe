"""The multi-replica host logic of bench.py on CPU: two ranks on the gloo
backend (the layer itself is single-GPU; N GPUs run N independent replicas
whose timing is the slowest rank's).  Each rank reports a different time;
both must see the maximum, and the whole-job throughput must count every
rank's tokens over that time.  The reference arm under torchrun runs on
rank 0 only: any other rank returns at once without output."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.reduce_max(10.0 + 5.0 * rank, world, "cpu")
        out[rank] = (ms, bench.job_tokens_per_s(world, 16384, 200, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_is_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for ms, v in res.values():
        assert ms == 15.0
        assert v == pytest.approx(2 * 16384 * 200 / 15e-3, rel=1e-12)


def test_single_rank_needs_no_process_group():
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_max(3.25, 1, "cpu") == 3.25
    assert bench.job_tokens_per_s(1, 1000, 10, 2.0) == pytest.approx(5e6)


def test_reference_arm_other_ranks_do_nothing(monkeypatch):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload="e64_bf16", steps=2, warmup=1)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args) is None
    assert buf.getvalue() == ""
