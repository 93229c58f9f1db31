"""Tensor parallelism of the fused KDA block over heads.

"KDA Block TKG Kernel API Reference": each rank runs the block on its own
num_head heads (Dimensions: num_head is the per-rank head count, a multiple
of the head group), with W_in's g_a and f_a columns replicated on every rank
(:param W_in:), and its `out` is this rank's partial of the output projection
until the caller reduces it across the tensor-parallel group (:param out:).

This module is the host side of that: it cuts the block's parameters and
state into per-rank shards (done once, when weights are loaded: index
gathers on the device, no arithmetic) and sums the ranks' partial `out` with
torch.distributed.  Every step of the block itself runs in libkda's kernels
(kda_block_tkg on the shard).

Per rank r of tp, heads h0 = r * nh / tp .. h0 + nh / tp - 1 (nh_r of them):

  sharded by head     W_in q, k columns (channel-outer: column d * nh + h),
                      W_in v columns (head-outer: h * V + d), W_in beta
                      columns (h), W_fb columns (head-outer), W_gb columns
                      (channel-outer), conv_w and conv_state channels (q, k
                      channel-outer, v head-outer), A_log, dt_bias columns,
                      W_o rows (head-outer), S heads
  replicated          gamma_in, W_in g_a and f_a columns, gamma_o, hidden

Each shard is laid out exactly like a whole block with nh_r heads (local head
hl = h - h0), so kda_block_tkg runs on it unchanged; sum over ranks of the
shards' `out` is the whole block's `out`.
"""
from __future__ import annotations

import torch

BLOCK_PARAMS = ("gamma_in", "W_in", "W_fb", "W_gb", "conv_w", "A_log", "dt_bias", "gamma_o",
                "W_o")


def head_range(nh: int, tp: int, rank: int) -> tuple[int, int]:
    if tp < 1 or nh % tp != 0 or not 0 <= rank < tp:
        raise ValueError(f"{nh} heads do not split over tp = {tp} (rank {rank})")
    nh_r = nh // tp
    return rank * nh_r, nh_r


def channel_outer(nh: int, width: int, h0: int, nh_r: int, device=None) -> torch.Tensor:
    """Global indices, in local order d * nh_r + hl, of the channel-outer
    columns d * nh + h of heads h0 .. h0 + nh_r - 1 (d < width)."""
    d = torch.arange(width, device=device)[:, None]
    h = torch.arange(h0, h0 + nh_r, device=device)[None, :]
    return (d * nh + h).reshape(-1)


def head_outer(width: int, h0: int, nh_r: int, device=None) -> torch.Tensor:
    """Global indices of the head-outer columns h * width + d of the shard."""
    return torch.arange(h0 * width, (h0 + nh_r) * width, device=device)


def _dims(W_fb: torch.Tensor, W_gb: torch.Tensor, A_log: torch.Tensor):
    nh = A_log.numel()
    K = W_fb.shape[0]
    V = W_gb.shape[1] // nh
    return nh, K, V


def shard_block_params(p: dict, tp: int, rank: int) -> dict:
    """This rank's block parameters (keys BLOCK_PARAMS), laid out as a whole
    block with nh / tp heads."""
    nh, K, V = _dims(p["W_fb"], p["W_gb"], p["A_log"])
    h0, nh_r = head_range(nh, tp, rank)
    dev = p["W_in"].device
    CQ, CV = K * nh, V * nh
    q_cols = channel_outer(nh, K, h0, nh_r, dev)
    v_cols = head_outer(V, h0, nh_r, dev)
    off_ga = 2 * CQ + CV
    cols = torch.cat([
        q_cols,                                                  # q
        CQ + q_cols,                                             # k
        2 * CQ + v_cols,                                         # v
        torch.arange(off_ga, off_ga + K, device=dev),            # g_a (replicated)
        off_ga + K + torch.arange(h0, h0 + nh_r, device=dev),    # beta
        torch.arange(off_ga + K + nh, off_ga + 2 * K + nh, device=dev),  # f_a (replicated)
    ])
    conv_idx = [q_cols, q_cols, v_cols]  # per stream: q, k channel-outer; v head-outer
    conv_w = torch.stack([p["conv_w"][s].index_select(-1, conv_idx[s]) for s in range(3)])
    return {
        "gamma_in": p["gamma_in"],
        "W_in": p["W_in"].index_select(1, cols).contiguous(),
        "W_fb": p["W_fb"].index_select(1, head_outer(K, h0, nh_r, dev)).contiguous(),
        "W_gb": p["W_gb"].index_select(1, channel_outer(nh, V, h0, nh_r, dev)).contiguous(),
        "conv_w": conv_w.contiguous(),
        "A_log": p["A_log"].reshape(1, nh)[:, h0:h0 + nh_r].contiguous(),
        "dt_bias": p["dt_bias"][:, h0:h0 + nh_r].contiguous(),
        "gamma_o": p["gamma_o"],
        "W_o": p["W_o"][h0 * V:(h0 + nh_r) * V].contiguous(),
    }


def shard_block_state(S: torch.Tensor, conv_state: torch.Tensor, tp: int, rank: int):
    """This rank's S [B, nh_r, K, V] and conv_state [B, 3, K * nh_r, Kc - 1]."""
    B, nh, K, V = S.shape
    h0, nh_r = head_range(nh, tp, rank)
    dev = S.device
    idx = [channel_outer(nh, K, h0, nh_r, dev), channel_outer(nh, K, h0, nh_r, dev),
           head_outer(V, h0, nh_r, dev)]
    cs = torch.stack([conv_state[:, s].index_select(1, idx[s]) for s in range(3)], dim=1)
    return S[:, h0:h0 + nh_r].contiguous(), cs.contiguous()


def gather_block_state(S_shards, cs_shards):
    """Inverse of shard_block_state over all ranks (shards in rank order)."""
    tp = len(S_shards)
    S = torch.cat(list(S_shards), dim=1)
    B, nh, K, V = S.shape
    Kc1 = cs_shards[0].shape[-1]
    cs = torch.empty((B, 3, K * nh, Kc1), dtype=cs_shards[0].dtype, device=cs_shards[0].device)
    for r, part in enumerate(cs_shards):
        h0, nh_r = head_range(nh, tp, r)
        idx = [channel_outer(nh, K, h0, nh_r, cs.device), channel_outer(nh, K, h0, nh_r, cs.device),
               head_outer(V, h0, nh_r, cs.device)]
        for s in range(3):
            cs[:, s].index_copy_(1, idx[s], part[:, s])
    return S, cs


def reduce_partial_out(out: torch.Tensor, group=None) -> torch.Tensor:
    """Sum this rank's partial `out` over the tensor-parallel group, in place
    (torch.distributed all-reduce: NCCL for CUDA tensors, gloo on the CPU)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    return out


def kda_block_tkg_tp(out, hidden, shard: dict, S, conv_state, scale, lower_bound,
                     rms_norm_eps=1e-5, l2_eps=1e-6, group=None, **kw):
    """One tensor-parallel block step on this rank: kda_block_tkg on the
    rank's shard (`shard` from shard_block_params; S and conv_state from
    shard_block_state, advanced in place), then the all-reduce of `out`
    over the group.  Returns the status word of the local call."""
    from . import kda_block_tkg
    status = kda_block_tkg(out, hidden, *[shard[k] for k in BLOCK_PARAMS], S, conv_state, scale,
                           lower_bound, rms_norm_eps, l2_eps, **kw)
    reduce_partial_out(out, group)
    return status
