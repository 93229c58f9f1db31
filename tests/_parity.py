"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding, run the float64 oracle on the same inputs (or on a sample of the
requests), and compare within the stated tolerances:

  outputs   max |gpu - ref| <= 1e-3 * (1 + |ref|)   element by element
  state     ||gpu - ref||_F / ||ref||_F <= 1e-5      per advanced state tile
  slots     untouched slots bit-identical; status words exact
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


def to_device(inp: dict, dev="cuda") -> dict:
    d = {}
    for key, val in inp.items():
        d[key] = val.to(dev) if isinstance(val, torch.Tensor) else val
    return d


def gpu_decode(inp: dict, dev="cuda", output_fill=float("nan")):
    """Run kda_decode on a copy of the pool; returns (output, pool, status)."""
    d = to_device(inp, dev)
    out = torch.full((inp["T"], inp["HV"], inp["V"]), output_fill, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kda_decode(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
               d["dt_bias"], d["cu_seqlens"], d["state_pool"], d["state_indices"],
               gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"], dev_status=status)
    torch.cuda.synchronize()
    return out, d["state_pool"], int(status.item())


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
