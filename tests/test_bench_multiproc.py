"""bench.py's N > 1 path (independent replicas, one per GPU) on CPU with
two gloo ranks: the slowest rank's time and the sum of all ranks' tokens
make the whole-job throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_setup()
    assert (w, r, lr) == (world, rank, rank)
    local_ms = 100.0 + 50.0 * rank          # rank 1 is the slow one
    local_tokens = 16 * 1024 * 50
    bench.barrier(world)
    ms, tokens, value = bench.aggregate(local_ms, local_tokens, world)
    out.put((rank, ms, tokens, value))
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, tokens, value in res:
        assert ms == 150.0                    # max over ranks
        assert tokens == 2 * 16 * 1024 * 50   # sum over ranks
        assert abs(value - tokens / 0.150) < 1e-6 * value
