"""The benchmark's multi-rank path on CPU: two gloo ranks in spawned processes.

Every rank serves its own sequences (its own seed) and the ranks meet only at a barrier and
at the max-over-ranks step time; the reference arm runs on rank 0 alone.  These are the host
steps of a multi-GPU run; each rank's GPU work is the single-GPU path the GPU tests cover.
"""
import argparse
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        ms = bench.max_over_ranks(1.0 + 0.5 * rank, w, "cpu")     # rank 1 is the slower one
        value = bench.job_value(32, w, ms)
        # the reference arm: ranks other than 0 return without work
        ref = bench.run_reference(argparse.Namespace(steps=1, warmup=0), rank, w) if rank != 0 else "rank 0"
        q.put((rank, r, w, local, ms, value, bench.rank_seed(1, rank), ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    seeds = set()
    for rank, r, w, local, ms, value, seed, ref in results:
        assert (r, w, local) == (rank, 2, rank)
        assert ms == 1.5                                   # the slowest rank's time, on every rank
        assert value == 32 * 2 / 1.5e-3                    # all ranks' queries over that time
        seeds.add(seed)
        if rank != 0:
            assert ref is None
    assert len(seeds) == 2                                 # independent sequences per rank
