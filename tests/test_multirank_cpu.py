"""The N > 1 path of bench.py on CPU: two gloo ranks exercise the barrier, the
max-over-ranks timing, the whole-job rate and the rank-0-only reference arm.
The path shards as independent replicas (one per GPU), so these host steps
are all the multi-rank logic there is."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        cpu = torch.device("cpu")
        bench.barrier(world)
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, world, cpu)
        rate = bench.whole_job_rate(1000.0, ms_max, world)

        class Args:
            workload, steps, warmup = "qwen3_8b_l1", 1, 0

        ref = bench.run_reference(Args, rank, world) if rank == 1 else "skipped"
        out.put((rank, ms_max, rate, bench.replica_seed(rank), ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_by_the_slowest_and_scale_weakly():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r, ms_max, rate, seed, ref = q.get(timeout=120)
        res[r] = (ms_max, rate, seed, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 15.0            # max over ranks, seen by every rank
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1000.0 / 0.015)   # all ranks' units / slowest time
    assert res[0][2] != res[1][2]                    # independent replicas
    assert res[1][3] is None                         # the reference arm runs on rank 0 only
