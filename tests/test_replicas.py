"""The multi-GPU path of bench.py is replicas only: every rank runs the whole
layer on its own GPU and the ranks meet only to time the job (a barrier on both
sides of the timed region, the slowest rank's time, the sum of the tokens).
This covers that plumbing with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist()
    assert (d.world, d.rank) == (world, rank)
    d.barrier()
    slowest = d.reduce(10.0 + rank, "max")  # per-rank step time: the job takes the slowest
    tokens = d.reduce(100.0 * (rank + 1), "sum")  # whole-job tokens: every rank's units
    d.barrier()
    d.close()
    out.put((rank, slowest, tokens))


@pytest.mark.timeout(120)
def test_replica_timing_plumbing_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    results = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slowest, tokens in results:
        assert slowest == 11.0
        assert tokens == 300.0


def test_single_process_is_world_one():
    sys.path.insert(0, ROOT)
    import bench

    old = {k: os.environ.pop(k, None) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    try:
        d = bench.Dist()
        assert d.world == 1 and d.rank == 0 and d.dist is None
        assert d.reduce(3.5, "max") == 3.5
    finally:
        for k, v in old.items():
            if v is not None:
                os.environ[k] = v
