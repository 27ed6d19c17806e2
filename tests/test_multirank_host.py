"""The multi-rank (weak-scaling) path of bench.py on the CPU, with two gloo ranks: every rank
times its own full workload, the job takes the slowest rank's times, and the whole-job
throughput counts every rank's tokens. The path exchanges no data between ranks (the
(batch row, kv head) groups are independent); the only collective is this maximum."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local = [10.0 + rank, 5.0 * (world - rank), 1.0 + 0.25 * rank]
        got = bench.max_over_ranks(local, "cpu", world)
        q.put((rank, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in procs:
            rank, got = q.get(timeout=120)
            results[rank] = got
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    # rank 0 sent [10, 10, 1], rank 1 [11, 5, 1.25]: both hold the element-wise maximum
    assert results[0] == results[1] == [11.0, 10.0, 1.25]


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 1.5], "cpu", 1) == [3.0, 1.5]


def test_whole_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(2048, 1, 1.0) == pytest.approx(2.048e6)
    assert bench.job_throughput(2048, 8, 1.0) == pytest.approx(8 * 2.048e6)
    assert bench.job_throughput(2048, 8, 2.0) == pytest.approx(4 * 2.048e6)
