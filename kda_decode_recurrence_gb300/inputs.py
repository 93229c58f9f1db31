"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and arranges them in the documented
shapes and dtypes; it holds none of the method's arithmetic.  Both the CUDA
path's tests/benchmark and the float64 oracle consume what it returns, which is
why it lives apart from both.

Draws use numpy's PCG64 (``numpy.random.default_rng(seed)``) in the order
listed in each function; bf16 tensors are the fp32 draws rounded to nearest
even (torch's float32 -> bfloat16 conversion).  Everything is returned as CPU
torch tensors; callers move them to the device.

Workloads (sizes from the decode and block API pages: 96 heads, dk = dv = 128,
conv taps 4, gate lower bound -5, eps 1e-5 / 1e-6):

  tiny        B=2 (3 and 5 tokens), H=HV=4, pool [8, 4, 128, 128] N(0, 0.1),
              softplus gate, seed 0
  single      B=64 x 1 token, H=HV=96, pool [256, 96, 128, 128] N(0, 0.05),
              softplus gate, seed 1
  grouped     B=256 x 1 token, H=48, HV=96 (G=2), pool [512, 96, 128, 128]
              N(0, 0.05), softplus gate, seed 2
  varlen      B=64, 1..8 tokens each, H=HV=96, pool [128, 96, 128, 128]
              N(0, 0.05), lower-bound gate (-5), seed 3
  block       B=32, n=1, Hd=4096, nh=32, K=V=128, Kc=4, seed 4
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

GATE_SOFTPLUS = 0
GATE_LOWER_BOUND = 1


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    H: int
    HV: int
    max_slots: int
    pool_std: float
    gate_mode: int
    seed: int
    lengths: tuple | None = None      # fixed per-request token counts
    tokens_per_request: int = 1       # used when lengths is None and not varlen
    varlen_max: int = 0               # >0: lengths drawn uniform in 1..varlen_max
    lower_bound: float = -5.0
    K: int = 128
    V: int = 128


DECODE_CONFIGS = {
    "tiny": DecodeConfig("tiny", B=2, H=4, HV=4, max_slots=8, pool_std=0.1,
                         gate_mode=GATE_SOFTPLUS, seed=0, lengths=(3, 5)),
    "single": DecodeConfig("single", B=64, H=96, HV=96, max_slots=256, pool_std=0.05,
                           gate_mode=GATE_SOFTPLUS, seed=1),
    "grouped": DecodeConfig("grouped", B=256, H=48, HV=96, max_slots=512, pool_std=0.05,
                            gate_mode=GATE_SOFTPLUS, seed=2),
    "varlen": DecodeConfig("varlen", B=64, H=96, HV=96, max_slots=128, pool_std=0.05,
                           gate_mode=GATE_LOWER_BOUND, seed=3, varlen_max=8),
}


@dataclass(frozen=True)
class BlockConfig:
    name: str = "block"
    B: int = 32
    n: int = 1
    Hd: int = 4096
    nh: int = 32
    K: int = 128
    V: int = 128
    Kc: int = 4
    weight_std: float = 0.02
    state_std: float = 0.05
    lower_bound: float = -5.0
    rms_norm_eps: float = 1e-5
    l2_eps: float = 1e-6
    seed: int = 4


BLOCK_CONFIG = BlockConfig()


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _f32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))


def _normal(rng, shape, std=1.0) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def decode_inputs(cfg: DecodeConfig | str, *, seed: int | None = None,
                  B: int | None = None, H: int | None = None, HV: int | None = None,
                  max_slots: int | None = None, lengths=None) -> dict:
    """Draw one decode workload.  Keyword overrides shrink a config for tests.

    Draw order: lengths (varlen only), q, k, v, raw_gate, beta_logits, a_log,
    dt_bias, state_pool, state_indices.
    """
    if isinstance(cfg, str):
        cfg = DECODE_CONFIGS[cfg]
    B = cfg.B if B is None else B
    H = cfg.H if H is None else H
    HV = cfg.HV if HV is None else HV
    N = cfg.max_slots if max_slots is None else max_slots
    K, V = cfg.K, cfg.V
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    if lengths is None:
        if cfg.varlen_max > 0:
            lengths = rng.integers(1, cfg.varlen_max + 1, size=B)
        elif cfg.lengths is not None:
            lengths = np.asarray(cfg.lengths)
        else:
            lengths = np.full(B, cfg.tokens_per_request)
    lengths = np.asarray(lengths, dtype=np.int64)
    assert lengths.shape == (B,)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    q = _bf16(_normal(rng, (T, H, K)))
    k = _bf16(_normal(rng, (T, H, K)))
    v = _bf16(_normal(rng, (T, HV, V)))
    raw_gate = _f32(_normal(rng, (T, HV, K)))
    beta_logits = _f32(_normal(rng, (T, HV)))
    a_log = _f32(np.log(rng.uniform(1.0, 16.0, size=HV)))
    dt_bias = _f32(_normal(rng, (HV, K), 0.1))
    state_pool = _f32(_normal(rng, (N, HV, K, V), cfg.pool_std))
    state_indices = torch.from_numpy(rng.permutation(N)[:B].astype(np.int32))
    return {
        "q": q, "k": k, "v": v, "raw_gate": raw_gate, "beta_logits": beta_logits,
        "a_log": a_log, "dt_bias": dt_bias,
        "cu_seqlens": torch.from_numpy(cu), "state_pool": state_pool,
        "state_indices": state_indices,
        "gate_mode": cfg.gate_mode, "lower_bound": cfg.lower_bound,
        "B": B, "T": T, "H": H, "HV": HV, "K": K, "V": V, "max_slots": N,
    }


def block_inputs(cfg: BlockConfig | None = None, *, seed: int | None = None, **overrides) -> dict:
    """Draw one fused-block workload (weights laid out as the block API page
    states them).  Draw order: hidden, W_in, W_fb, W_gb, conv_w, A_log,
    dt_bias, W_o, S, conv_state.  gamma_in and gamma_o are ones."""
    cfg = cfg or BLOCK_CONFIG
    if overrides:
        cfg = BlockConfig(**{**cfg.__dict__, **overrides})
    B, n, Hd, nh, K, V, Kc = cfg.B, cfg.n, cfg.Hd, cfg.nh, cfg.K, cfg.V, cfg.Kc
    I = 2 * K * nh + V * nh + 2 * K + nh
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    ws = cfg.weight_std
    hidden = _f32(_normal(rng, (B, n, Hd)))
    W_in = _bf16(_normal(rng, (Hd, I), ws))
    W_fb = _bf16(_normal(rng, (K, K * nh), ws))
    W_gb = _bf16(_normal(rng, (K, V * nh), ws))
    conv_w = _bf16(_normal(rng, (3, Kc, K * nh), ws))
    A_log = _f32(np.log(rng.uniform(1.0, 16.0, size=(1, nh))))
    dt_bias = _f32(_normal(rng, (K, nh), 0.1))
    W_o = _bf16(_normal(rng, (V * nh, Hd), ws))
    S = _f32(_normal(rng, (B, nh, K, V), cfg.state_std))
    conv_state = _f32(_normal(rng, (B, 3, K * nh, Kc - 1), cfg.state_std))
    return {
        "hidden": hidden, "gamma_in": torch.ones(1, Hd), "W_in": W_in, "W_fb": W_fb,
        "W_gb": W_gb, "conv_w": conv_w, "A_log": A_log, "dt_bias": dt_bias,
        "gamma_o": torch.ones(1, V), "W_o": W_o, "S": S, "conv_state": conv_state,
        "scale": K ** -0.5, "lower_bound": cfg.lower_bound,
        "rms_norm_eps": cfg.rms_norm_eps, "l2_eps": cfg.l2_eps,
        "B": B, "n": n, "Hd": Hd, "nh": nh, "K": K, "V": V, "Kc": Kc, "I": I,
    }


def to_f64(t) -> np.ndarray:
    """Widen a CPU tensor (bf16/fp32) to a float64 numpy array, exactly."""
    return t.detach().to("cpu").double().numpy()
