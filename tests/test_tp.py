"""Tensor parallelism of the fused block ("KDA Block TKG Kernel API
Reference", :param W_in: -- g_a and f_a replicated; :param out: -- each
rank's out is a partial until reduced across the group; Dimensions --
num_head per rank), host side, no GPU:

  * the float64 oracle run on each rank's shard gives partial outs whose sum
    is the oracle's whole block, and shard states that gather back into the
    whole block's advanced state (tp = 2 and 4, one and two tokens);
  * two gloo ranks, each with its own shard, reduce their partials with the
    library's all-reduce and both hold the whole block's out.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from kda_decode_recurrence_gb300 import tp

NAMES = tp.BLOCK_PARAMS


def small_block(seed, B=2, n=1, Hd=16, nh=4, K=4, Kc=4):
    rng = np.random.default_rng(seed)
    V = K
    I = 2 * K * nh + V * nh + 2 * K + nh
    p = dict(
        gamma_in=rng.uniform(0.5, 1.5, (1, Hd)), W_in=0.3 * rng.standard_normal((Hd, I)),
        W_fb=0.3 * rng.standard_normal((K, K * nh)), W_gb=0.3 * rng.standard_normal((K, V * nh)),
        conv_w=0.5 * rng.standard_normal((3, Kc, K * nh)),
        A_log=np.log(rng.uniform(1, 16, (1, nh))), dt_bias=0.1 * rng.standard_normal((K, nh)),
        gamma_o=rng.uniform(0.5, 1.5, (1, V)), W_o=0.3 * rng.standard_normal((V * nh, Hd)))
    state = dict(hidden=rng.standard_normal((B, n, Hd)),
                 S=0.1 * rng.standard_normal((B, nh, K, V)),
                 conv_state=0.5 * rng.standard_normal((B, 3, K * nh, Kc - 1)))
    return {k: torch.from_numpy(v) for k, v in p.items()}, {k: torch.from_numpy(v) for k, v in state.items()}


def run_oracle(p, hidden, S, cs):
    return oracle.kda_block_tkg(hidden.numpy(), *[p[k].numpy() for k in NAMES], S.numpy(),
                                cs.numpy(), scale=0.5, lower_bound=-5.0)


def shard_partial(p, st, tp_size, rank):
    shard = tp.shard_block_params(p, tp_size, rank)
    S_r, cs_r = tp.shard_block_state(st["S"], st["conv_state"], tp_size, rank)
    out, S_new, cs_new = run_oracle(shard, st["hidden"], S_r, cs_r)
    return out, torch.from_numpy(S_new), torch.from_numpy(cs_new)


@pytest.mark.parametrize("tp_size", [2, 4])
@pytest.mark.parametrize("n", [1, 2])
def test_shard_partials_sum_to_the_whole_block(tp_size, n):
    p, st = small_block(200 + tp_size + n, n=n)
    out, S_new, cs_new = run_oracle(p, st["hidden"], st["S"], st["conv_state"])
    parts = [shard_partial(p, st, tp_size, r) for r in range(tp_size)]
    np.testing.assert_allclose(sum(o for o, _, _ in parts), out, rtol=0, atol=1e-12)
    S_g, cs_g = tp.gather_block_state([s for _, s, _ in parts], [c for _, _, c in parts])
    np.testing.assert_array_equal(S_g.numpy(), S_new)      # each head's update is local
    np.testing.assert_array_equal(cs_g.numpy(), cs_new)
    # no single shard carries the whole output
    assert all(np.abs(o - out).max() > 1e-3 for o, _, _ in parts)


def test_one_rank_shard_is_the_whole_block():
    p, st = small_block(210)
    shard = tp.shard_block_params(p, 1, 0)
    for k in NAMES:
        assert torch.equal(shard[k].reshape(p[k].shape), p[k]), k
    S_r, cs_r = tp.shard_block_state(st["S"], st["conv_state"], 1, 0)
    assert torch.equal(S_r, st["S"]) and torch.equal(cs_r, st["conv_state"])


def test_shards_cover_every_head_channel_once():
    nh, K, tp_size = 8, 4, 4
    cols = torch.cat([tp.channel_outer(nh, K, *tp.head_range(nh, tp_size, r)) for r in range(tp_size)])
    assert sorted(cols.tolist()) == list(range(nh * K))
    cols = torch.cat([tp.head_outer(K, *tp.head_range(nh, tp_size, r)) for r in range(tp_size)])
    assert cols.tolist() == list(range(nh * K))
    with pytest.raises(ValueError):
        tp.head_range(12, 5, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p, st = small_block(220)
        partial, _, _ = shard_partial(p, st, world, rank)
        out = torch.from_numpy(partial.copy())
        tp.reduce_partial_out(out)
        q.put((rank, out.numpy(), partial))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_all_reduce_the_partial_outs():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda x: x[0])
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    p, st = small_block(220)
    whole, _, _ = run_oracle(p, st["hidden"], st["S"], st["conv_state"])
    for rank, reduced, partial in res:
        np.testing.assert_allclose(reduced, whole, rtol=0, atol=1e-12)
        assert np.abs(partial - whole).max() > 1e-3
