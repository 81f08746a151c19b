"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2).

The decode path shards as independent replicas (each rank owns its own
streams; no collective on the data path). What ranks share is the timing
reduction: the job's time is the slowest rank's, and the job's throughput is
the bytes of all ranks over that time.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(0.5 + rank, world)   # ranks report 0.5 s and 1.5 s
    bench.barrier(world)
    q.put((rank, t))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=100) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert got == {0: 1.5, 1: 1.5}


def test_single_rank_accounting():
    import bench
    total, tokens, per_kind = bench.step_accounting(64, 4096)
    # 21 sliding layers of 511 cached tokens and 7 full layers of 4096, 2 KV heads x 256 dims
    assert per_kind["sliding"][0] == 64 * 511 * 2048
    assert per_kind["full"][0] == 64 * 4096 * 2048
    assert tokens == 64 * (21 * 512 + 7 * 4097)
    assert total > 21 * per_kind["sliding"][0] + 7 * per_kind["full"][0]
