"""Host logic of the N > 1 benchmark path on CPU with gloo, world size 2:
each rank draws its own batch (weak scaling, no data-path collective) and
the job time is the maximum over ranks."""
import os
import socket

import pytest
import torch
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
        t = bench.max_over_ranks(1.0 + rank, world)
        seed = bench.shard_seed(2, rank)
        from kda_decode_recurrence_gb300.inputs import decode_inputs
        inp = decode_inputs("grouped", B=2, H=2, HV=4, max_slots=4, seed=seed)
        bench.barrier(world)
        q.put((rank, t, seed, float(inp["state_pool"].sum())))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_max_and_shards():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]            # max over ranks on every rank
    assert res[0][2] != res[1][2]                        # distinct per-rank batches
    assert res[0][3] != res[1][3]
