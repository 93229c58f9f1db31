"""kda_block_tkg on the GPU (through the C ABI) against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from kda_decode_recurrence_gb300 import block_workspace_size, kda_block_tkg
from kda_decode_recurrence_gb300.inputs import block_inputs, to_f64

from _parity import assert_outputs_close, assert_states_close, to_device

pytestmark = pytest.mark.gpu

WEIGHTS = ("hidden", "gamma_in", "W_in", "W_fb", "W_gb", "conv_w", "A_log", "dt_bias",
           "gamma_o", "W_o")


def gpu_block(inp, workspace=None):
    d = to_device(inp)
    out = torch.full((inp["B"], inp["n"], inp["Hd"]), float("nan"), device="cuda")
    kda_block_tkg(out, *[d[k] for k in WEIGHTS], d["S"], d["conv_state"], inp["scale"],
                  inp["lower_bound"], inp["rms_norm_eps"], inp["l2_eps"], workspace=workspace)
    torch.cuda.synchronize()
    return out, d["S"], d["conv_state"]


def oracle_block(inp):
    return oracle.kda_block_tkg(*[to_f64(inp[k]) for k in WEIGHTS], to_f64(inp["S"]),
                                to_f64(inp["conv_state"]), inp["scale"], inp["lower_bound"],
                                inp["rms_norm_eps"], inp["l2_eps"])


def check_block(inp):
    out, S, cs = gpu_block(inp)
    ref_out, ref_S, ref_cs = oracle_block(inp)
    assert_outputs_close(out.cpu().numpy(), ref_out, "out")
    assert_states_close(S.cpu().numpy(), ref_S, "S")
    # conv_state: the shifted entries are copies, the newest is the projection
    cs = cs.cpu().numpy()
    np.testing.assert_array_equal(cs[..., :-1], to_f64(inp["conv_state"])[..., 1:])
    assert_outputs_close(cs[..., -1], ref_cs[..., -1], "conv_state")


def test_block_full_config():
    check_block(block_inputs())


@pytest.mark.parametrize("B,Hd,nh,Kc", [(37, 256, 8, 4), (3, 384, 16, 3), (1, 128, 8, 2)])
def test_block_small_and_ragged(B, Hd, nh, Kc):
    check_block(block_inputs(B=B, Hd=Hd, nh=nh, Kc=Kc, seed=60 + B))


def test_block_workspace_reuse_is_stateless():
    inp = block_inputs(B=5, Hd=256, nh=8, seed=70)
    ws = torch.full((block_workspace_size(5, 1, 256, 8, 128, 128, 4),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    out1, _, _ = gpu_block(inp, ws)
    out2, _, _ = gpu_block(inp, ws)       # stale workspace contents must not matter
    assert torch.equal(out1, out2)
