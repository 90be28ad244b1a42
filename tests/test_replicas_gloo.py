"""Multi-GPU layout of the benchmark: independent replicas, no data-path
collective; only the timing is reduced (max over ranks). Checked with two
gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
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
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        elapsed = 1.5 + rank                      # each replica times its own steps
        mx = bench.reduce_max(elapsed, world)
        bench.barrier(world)
        q.put((rank, mx))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_replica_seeds_differ():
    import synth
    a = synth.workload("qwen7b_b1")
    b = a.with_(seed=a.seed + 1000)
    assert a.seed != b.seed
