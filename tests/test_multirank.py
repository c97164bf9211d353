"""Host-side logic of the N-replica benchmark on CPU with gloo, world size 2.

The path shards by replicas only (each GPU runs the whole workload on its own
prompts; no data-path collective).  What is shared across ranks is timing:
a barrier around the timed region, the MAX of the ranks' times, and the
whole-job throughput = the work every rank did, summed, over the slowest
time.  These run here on CPU, together with the inputs each replica draws:
the same weight on every rank (one model) and its own prompts.
"""
import hashlib
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import workloads
        bench.barrier(world)
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        mx = bench.allreduce_max(local_ms, world)
        agg = bench.aggregate_tflops((rank + 1) * 10 ** 12, mx, world)   # each rank counts its own work
        env = bench.dist_env()
        mine = workloads.for_replica(bench.CFG, rank)
        digests = [None] * world
        dist.all_gather_object(digests, (
            hashlib.sha256(workloads.bits(workloads.make_activation(mine)).tobytes()).hexdigest(),
            hashlib.sha256(workloads.bits(workloads.make_weight(mine)).tobytes()).hexdigest()))
        # the reference arm: only rank 0 works and prints; rank 1 returns at once
        class A:
            steps, warmup, gpus = 1, 3, world
        rc = bench.run_reference(A) if rank == 1 else 0
        q.put((rank, mx, agg, env, rc, digests))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_aggregation():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, agg, env, rc, digests in results:
        assert mx == 15.0                               # max over ranks
        assert agg == pytest.approx((1 + 2) * 1e12 / 15e-3 / 1e12)
        assert env == (2, rank, rank)
        assert rc == 0
        (x0, w0), (x1, w1) = digests
        assert x0 != x1                                 # each replica runs its own prompts
        assert w0 == w1                                 # of the one shared model
