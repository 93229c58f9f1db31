"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding, run the float64 oracle on the same inputs (or on a sample of the
requests), and compare within the stated tolerances:

  outputs   max |gpu - ref| <= 1e-3 * (1 + |ref|)   element by element
  state     ||gpu - ref||_F / ||ref||_F <= 1e-5      per advanced state tile
  slots     untouched slots bit-identical; status words exact
  bounds    every buffer a kernel writes sits between two guard regions
            filled with a byte pattern, checked unchanged after the call
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kda_decode_recurrence_gb300 import kda_decode
from kda_decode_recurrence_gb300.inputs import to_f64

OUT_ATOL = 1e-3
STATE_RTOL = 1e-5
TOKEN_KEYS = ("q", "k", "v", "raw_gate", "beta_logits")


GUARD_BYTES = 4096      # a multiple of 256, so the guarded tensor keeps its alignment
GUARD_PATTERN = 0xA5


class Guarded:
    """A device tensor with a guard region of GUARD_BYTES on each side, filled
    with GUARD_PATTERN; ``intact()`` reports whether a kernel wrote outside
    the tensor (a write past either end changes a guard byte).  Stands in
    for a bounds-checking tool on this device."""

    def __init__(self, shape, dtype, dev="cuda", fill=None, like: torch.Tensor | None = None):
        shape = tuple(shape)
        itemsize = torch.empty(0, dtype=dtype).element_size()
        nbytes = int(np.prod(shape, dtype=np.int64)) * itemsize
        self.raw = torch.empty(2 * GUARD_BYTES + nbytes, dtype=torch.uint8, device=dev)
        self.raw[:GUARD_BYTES].fill_(GUARD_PATTERN)
        self.raw[GUARD_BYTES + nbytes:].fill_(GUARD_PATTERN)
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
        if like is not None:
            self.t.copy_(like)
        elif fill is not None:
            self.t.fill_(fill)

    def intact(self) -> bool:
        return bool((self.raw[:GUARD_BYTES] == GUARD_PATTERN).all().item()) and bool(
            (self.raw[-GUARD_BYTES:] == GUARD_PATTERN).all().item())


def guarded_copy(t: torch.Tensor, dev="cuda") -> Guarded:
    return Guarded(t.shape, t.dtype, dev, like=t)


def to_device(inp: dict, dev="cuda") -> dict:
    d = {}
    for key, val in inp.items():
        d[key] = val.to(dev) if isinstance(val, torch.Tensor) else val
    return d


def gpu_decode(inp: dict, dev="cuda", output_fill=float("nan")):
    """Run kda_decode on a copy of the pool; returns (output, pool, status).
    The output and the pool are guarded; the guards are checked here."""
    d = to_device(inp, dev)
    out = Guarded((inp["T"], inp["HV"], inp["V"]), torch.float32, dev, fill=output_fill)
    pool = guarded_copy(inp["state_pool"], dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kda_decode(out.t, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
               d["dt_bias"], d["cu_seqlens"], pool.t, d["state_indices"],
               gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"], dev_status=status)
    torch.cuda.synchronize()
    assert out.intact(), "write outside output"
    assert pool.intact(), "write outside state_pool"
    return out.t, pool.t, int(status.item())


def oracle_decode_sample(inp: dict, bs) -> tuple:
    """The oracle on requests ``bs`` only (their tokens and their slots).
    Returns (token rows, slots, ref_out [rows, HV, V], ref_states [len(bs), HV, K, V])."""
    cu = inp["cu_seqlens"].numpy()
    idx = inp["state_indices"].numpy()
    bs = list(bs)
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in bs]).astype(np.int64)
    lengths = np.array([cu[b + 1] - cu[b] for b in bs])
    slots = idx[bs]
    assert np.all(slots >= 0)
    sub_pool = to_f64(inp["state_pool"][torch.from_numpy(slots.astype(np.int64))])
    tok = {key: to_f64(inp[key][torch.from_numpy(rows)]) for key in TOKEN_KEYS}
    out, pool, st = oracle.kda_decode(
        tok["q"], tok["k"], tok["v"], tok["raw_gate"], tok["beta_logits"], to_f64(inp["a_log"]),
        to_f64(inp["dt_bias"]), np.concatenate([[0], np.cumsum(lengths)]), sub_pool,
        np.arange(len(bs)), gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"])
    assert st == 0
    return rows, slots, out, pool


def assert_all_requests_match(inp: dict, out: torch.Tensor, pool: torch.Tensor, bs=None,
                              chunk: int = 32, out_bound=None):
    """Every request in ``bs`` (default: all with a valid slot) against the
    oracle: all of its token rows and all of its advanced tiles, ``chunk``
    requests at a time so the float64 copies stay small.  ``out`` [T, HV, V]
    and ``pool`` (K-first tiles) are device tensors.  ``out_bound(got, ref)``
    replaces the output check (e.g. for bf16 outputs)."""
    idx = inp["state_indices"].numpy()
    if bs is None:
        bs = [b for b in range(inp["B"]) if 0 <= idx[b] < inp["max_slots"]]
    bs = list(bs)
    for i in range(0, len(bs), chunk):
        part = bs[i:i + chunk]
        rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, part)
        got = out[torch.from_numpy(rows).to(out.device)].float().cpu().numpy()
        if out_bound is None:
            assert_outputs_close(got, ref_out)
        else:
            out_bound(got.astype(np.float64), ref_out)
        assert_states_close(pool[torch.from_numpy(slots.astype(np.int64)).to(pool.device)].cpu().numpy(),
                            ref_pool)
    return len(bs)


def assert_outputs_close(gpu: np.ndarray, ref: np.ndarray, what="output"):
    gpu = np.asarray(gpu, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    err = np.abs(gpu - ref)
    bound = OUT_ATOL * (1.0 + np.abs(ref))
    worst = np.max(err / bound) if err.size else 0.0
    assert worst <= 1.0, f"{what}: max err/bound = {worst:.3g} (max abs err {err.max():.3g})"
    return worst


def assert_states_close(gpu: np.ndarray, ref: np.ndarray, what="state", tol=STATE_RTOL):
    """Relative Frobenius error per [K, V] tile (last two axes) <= tol."""
    gpu = np.asarray(gpu, dtype=np.float64)
    K, V = ref.shape[-2:]
    g = gpu.reshape(-1, K * V)
    r = ref.reshape(-1, K * V)
    rel = np.linalg.norm(g - r, axis=1) / np.maximum(np.linalg.norm(r, axis=1), 1e-300)
    worst = rel.max() if rel.size else 0.0
    assert worst <= tol, f"{what}: worst relative Frobenius error {worst:.3g} (bound {tol:.3g})"
    return worst
