"""The replicas path of bench.py on CPU: two gloo ranks (no GPU).

Each rank reports its own step timings; the job's time is the slowest rank's, element by
element, and the job's throughput counts the tokens of every replica against it. The
reference arm runs on rank 0 only: the other ranks return without work.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 5.0 - 2 * rank, 0.25 * (rank + 1)]  # rank 0: 1, 5, .25; rank 1: 2, 3, .5
        got = bench.max_over_ranks(mine, torch.device("cpu"), world)
        ref_rank = bench.run_reference(_Args(), _tiny())
        q.put((rank, got, ref_rank is None))
    finally:
        dist.destroy_process_group()


class _Args:
    steps = 1
    warmup = 0


def _tiny():
    import moe_synth
    return moe_synth.WORKLOADS["tiny"]


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        rank, got, ref_none = q.get(timeout=120)
        out[rank] = (got, ref_none)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        assert out[rank][0] == [2.0, 5.0, 0.5]
    assert out[0][1] is False      # rank 0 times the oracle
    assert out[1][1] is True       # other ranks do no work


def test_single_rank_and_throughput():
    import bench
    assert bench.max_over_ranks([3.0, 1.5], None, 1) == [3.0, 1.5]
    # 4 replicas of 64 tokens, slowest step 0.5 ms -> 512000 tokens/s for the job
    assert bench.job_tokens_per_s(4, 64, 0.5) == pytest.approx(512000.0)
