"""The multi-process (torchrun) path of bench.py on CPU: two gloo ranks agree on the job
time (max over ranks) and run disjoint replica instances. No GPU is involved."""
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
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        bench.barrier(world)
        t = bench.max_over_ranks(10.0 + rank, world)
        q.put((rank, t, bench.rank_instances(rank, 48)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_disjoint_instances():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [t for _, t, _ in res] == [11.0, 11.0]          # slowest rank sets the time
    inst0, inst1 = res[0][2], res[1][2]
    assert not set(inst0) & set(inst1) and len(inst0) == len(inst1) == 48
