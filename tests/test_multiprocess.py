"""The N > 1 bench path on CPU with gloo, world size 2: replicas draw distinct
batches, the timed region is the slowest rank's, and the whole-job value
counts every rank's tokens.  The path has no data collective (replicas only)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.WORKLOADS["llama2-7b-layer"]
        ms = [12.5, 17.25][rank]
        t_max = bench.max_over_ranks(ms)
        value = bench.whole_job_value(w, world, 10, t_max)
        seed = bench.replica_seed(w, 0, rank)
        q.put((rank, t_max, value, seed, bench._dist_env()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = bench.WORKLOADS["llama2-7b-layer"]
    per_rank_tokens = bench._kv_tokens_per_step(w) * 10
    for rank, t_max, value, seed, env in out:
        assert t_max == 17.25                                   # the slowest rank's time
        assert abs(value - 2 * per_rank_tokens / 17.25e-3) < 1e-6 * value
        assert env == (2, rank, 0)
    assert out[0][3] != out[1][3]                               # distinct replica batches
    # per-rank tokens: 8 batch rows x 4 layers x sum over 64 decode calls of the attended tokens
    assert bench._kv_tokens_per_step(w) == 4 * 8 * sum(4096 + s for s in range(1, 65))
