"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The gated-prefill path shards over independent sequences, so N GPUs run N independent
replicas with no collective on the data path; the only cross-rank steps are the barrier and
the max-over-ranks of the step time. These tests run those steps as two gloo ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.cpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        dist.barrier()
        slowest = bench.reduce_max(times[rank], world)
        value = bench.aggregate(1000, world, slowest)
        seed = bench.replica_seed(1234, rank)
        out.put((rank, slowest, value, seed))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_weak_scaling_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [0.004, 0.005]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, value, _ in res:
        assert slowest == pytest.approx(0.005)             # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 1000 / 0.005)    # tokens of all ranks / slowest time
    assert res[0][3] != res[1][3]                           # each replica draws its own batch


def test_single_rank_helpers_need_no_process_group():
    import bench
    assert bench.reduce_max(0.25, 1) == 0.25
    assert bench.aggregate(33024, 1, 0.001) == pytest.approx(33024 / 0.001)
