"""The benchmark's multi-rank path on CPU (gloo, world size 2): replicas time
independently, the job's time is the max over ranks, throughput counts every
replica's tokens, and the reference arm's non-zero ranks exit without work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank * 5.0, 3.0 - rank]          # rank 1 slower in the first, faster in the second
        got = bench.max_over_ranks(mine, world)
        q.put((rank, got, bench.job_throughput(world, 32768, got[0] / 100)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_world2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, thr in res:
        assert got == [15.0, 3.0]
        assert thr == pytest.approx(2 * 32768 / (0.15 / 1e3))


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.job_throughput(1, 1000, 2.0) == pytest.approx(500000.0)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0


def test_reference_arm_line_small_workload(monkeypatch, capsys):
    # the oracle timed as the reference arm prints one JSON line with impl = reference
    import json
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1", "--workload", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["metric"] == bench.METRIC
