"""bench.py's multi-rank host logic on CPU: two gloo ranks (world size 2).

Under torchrun every rank times its own replica; the job's time is the
slowest rank's (a MAX all-reduce) and its throughput all ranks' tokens over
that time.  The reference arm runs on rank 0 alone."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, seconds, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.slowest_rank_seconds(seconds[rank], world)
        tps = bench.job_tokens_per_s(100, seconds[rank], world)
        results[rank] = (slow, tps)
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, seconds = 2, [0.5, 0.8]
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), seconds, results), nprocs=world,
                 join=True)
        got = dict(results)
    for rank in range(world):
        slow, tps = got[rank]
        assert slow == pytest.approx(0.8)
        assert tps == pytest.approx(100 * world / 0.8)   # all ranks' tokens over the slowest


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_seconds(0.25, 1) == 0.25
    assert bench.job_tokens_per_s(100, 0.25, 1) == pytest.approx(400.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"], env=env, capture_output=True,
                         text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""
