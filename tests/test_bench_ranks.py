"""Host logic of the multi-GPU bench (replicas only, no collective on the data path): two
ranks over gloo on the CPU agree on the slowest rank's step time and report the whole
job's rate; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    ms_local = [2.0, 3.5][rank]
    dist.barrier()
    out = bench.whole_job(dist, ms_local, 8, world, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out))


def test_two_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        ms_max, rate = res[r]
        assert ms_max == pytest.approx(3.5)
        assert rate == pytest.approx(2 * 8 / 3.5e-3)


def test_one_rank_needs_no_collective():
    import bench

    assert bench.whole_job(None, 4.0, 8, 1, "cpu") == (4.0, pytest.approx(2000.0))


def test_reference_arm_runs_on_rank_zero_only():
    import bench

    class A:
        workload = "decode_b1"
        steps = 1
        warmup = 0

    assert bench.run_reference(A(), 1, 2) is None
