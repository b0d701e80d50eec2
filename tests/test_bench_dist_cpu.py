"""The multi-rank logic of bench.py on CPU: two gloo ranks agree on the slowest
rank's time, the whole-job value counts every rank's units, and the reference
arm prints from rank 0 only. No GPU: under torchrun each rank times its own
replica of the workload (no collective on the data path), and only the timing
reduction crosses ranks."""
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
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slowest
        total = bench.max_over_ranks(local_ms)
        value = bench.whole_job_value(1000, 4, world, total)
        out.put((rank, total, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, total, value in got:
        assert total == 15.0
        # 2 ranks x 4 steps x 1000 units in 15 ms
        assert value == pytest.approx(2 * 4 * 1000 / 0.015)


def test_single_process_needs_no_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_value(10, 2, 1, 4.0) == pytest.approx(5000.0)


def test_reference_arm_prints_from_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(bench.argparse.Namespace(workload=2, steps=1, warmup=0))
    assert buf.getvalue() == ""
