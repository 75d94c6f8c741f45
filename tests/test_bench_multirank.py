"""The benchmark's multi-GPU host logic on CPU: two gloo ranks, each timing its own replica.
The whole-job number takes the slowest rank's time and every rank's rows."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    tmax, value = bench.aggregate_over_ranks(times[rank], world, 4096, 10, "cpu")
    dist.barrier()
    out_q.put((rank, tmax, value))
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_slowest_rank():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [2.0, 5.0]  # ms for 10 steps on each rank
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tmax, value in res:
        assert tmax == 5.0
        assert abs(value - 2 * 4096 * 10 / 5e-3) < 1e-6


def test_single_rank_aggregation_is_local():
    sys.path.insert(0, ROOT)
    import bench
    tmax, value = bench.aggregate_over_ranks(4.0, 1, 100, 20, "cpu")
    assert tmax == 4.0 and abs(value - 100 * 20 / 4e-3) < 1e-9


def test_reference_arm_other_ranks_do_no_work(tmp_path):
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
