"""The benchmark's multi-rank logic on CPU, world size 2 over gloo: the job
time is the max over ranks, the job throughput counts every rank's units,
and the reference arm runs on rank 0 only.  (The data path has no
collective: every rank processes its own prompt.)"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                       # rank 1 is the slow one
        max_ms = bench.max_over_ranks(ms, world)
        total = bench.sum_over_ranks(rank + 1, world)
        thr = bench.job_throughput(8192, world, max_ms)
        bench.barrier(world)
        q.put((rank, max_ms, total, thr))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, max_ms, total, thr in res:
        assert max_ms == 15.0
        assert total == 3.0
        assert thr == pytest.approx(2 * 8192 / 0.015)


def test_reference_arm_prints_on_rank_0_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "q8_0_tiny"])
    assert buf.getvalue() == ""


def test_reference_arm_line(monkeypatch):
    sys.path.insert(0, ROOT)
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "q8_0_tiny",
                    "--reference-rows", "4"])
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
