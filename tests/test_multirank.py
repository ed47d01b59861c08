"""bench.py's multi-rank bookkeeping with two gloo ranks on the CPU.

The path has no exchange between GPUs (all tp shards live on one device), so
N GPUs run N independent replicas; the only cross-rank work is the barrier and
the max-over-ranks time / sum-over-ranks tokens that bench.py reports.
"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, lr, w = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    bench.barrier(w)
    elapsed = 100.0 + 25.0 * rank          # rank 1 is the slowest
    tokens = 4096 * 20
    res = bench.reduce_over_ranks(elapsed, tokens, w)
    q.put((rank, res))
    dist.destroy_process_group()


def test_two_rank_replicas_reduce():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        elapsed_max, tokens_all = out[r]
        assert elapsed_max == 125.0
        assert tokens_all == 2 * 4096 * 20
    # whole-job throughput is total tokens over the slowest rank's time
    assert tokens_all / (elapsed_max / 1e3) == 2 * 4096 * 20 / 0.125


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_over_ranks(12.5, 77, 1) == (12.5, 77)
