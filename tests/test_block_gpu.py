"""kda_block_tkg on the GPU (through the C ABI) against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from kda_decode_recurrence_gb300 import block_workspace_size, kda_block_tkg
from kda_decode_recurrence_gb300.inputs import block_inputs, to_f64

from _parity import STATE_RTOL, assert_outputs_close, assert_states_close, to_device

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
    # Each token multiplies S by decay factors exp(g) whose fp32 rounding the
    # gate amplifies (|dg/dgraw| <= |lower_bound| * exp(A_log) / 4 = 20 here),
    # so the relative state error grows with the tokens chained in one call:
    # the 1e-5 bound holds per token, n * 1e-5 for n tokens.
    assert_states_close(S.cpu().numpy(), ref_S, "S", tol=STATE_RTOL * inp["n"])
    # conv_state: the last Kc-1 pre-convolution inputs.  With one token the
    # older entries are exact copies shifted by one; entries that come from
    # this call's projection carry the GEMM's rounding.
    cs = cs.cpu().numpy()
    assert_outputs_close(cs, ref_cs, "conv_state")
    if inp["n"] == 1:
        np.testing.assert_array_equal(cs[..., :-1], to_f64(inp["conv_state"])[..., 1:])


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
    # the output projection adds its contraction splits with fp32 atomics, so
    # repeated calls agree to rounding, not bit for bit
    assert_outputs_close(out2.cpu().numpy(), out1.cpu().double().numpy(), "repeat")


# -------------------------------------------- n > 1 tokens per request

@pytest.mark.parametrize("B,n,Hd,nh,Kc", [(3, 2, 256, 8, 4), (5, 5, 384, 16, 3), (2, 3, 128, 8, 2)])
def test_block_multi_token_small(B, n, Hd, nh, Kc):
    check_block(block_inputs(B=B, n=n, Hd=Hd, nh=nh, Kc=Kc, seed=80 + B + n))


def test_block_multi_token_kimi_k3_weights():
    # the full weight shapes (Hd 4096, 32 heads) with a 4-token window, 8 requests
    check_block(block_inputs(B=8, n=4, seed=85))


def test_block_n_tokens_equal_n_single_token_calls():
    inp = block_inputs(B=4, n=3, Hd=256, nh=8, seed=86)
    out_all, S_all, cs_all = gpu_block(inp)
    step = dict(inp)
    step["n"] = 1
    S, cs = inp["S"], inp["conv_state"]
    outs = []
    for j in range(3):
        step["hidden"] = inp["hidden"][:, j:j + 1].contiguous()
        step["S"], step["conv_state"] = S, cs
        o, S, cs = gpu_block(step)
        S, cs = S.cpu(), cs.cpu()
        outs.append(o)
    np.testing.assert_allclose(torch.cat(outs, 1).cpu().numpy(), out_all.cpu().numpy(),
                               rtol=1e-5, atol=1e-5)
    assert_states_close(S.numpy(), S_all.cpu().double().numpy(), "S")
    np.testing.assert_allclose(cs.numpy(), cs_all.cpu().numpy(), rtol=1e-6, atol=1e-7)


# Row blocks of more than 32 rows: the projection GEMMs take two 128-column
# weight tiles per CTA against each activation tile (one CTA per SM).
@pytest.mark.parametrize("B,n,Hd,nh,Kc", [(17, 4, 256, 8, 4), (9, 7, 384, 16, 3), (33, 1, 256, 8, 2)])
def test_block_row_blocks_over_32(B, n, Hd, nh, Kc):
    check_block(block_inputs(B=B, n=n, Hd=Hd, nh=nh, Kc=Kc, seed=90 + B + n))


def test_block_multi_token_full_shapes_128_rows():
    # the full weight shapes with B = 32 requests x 4 tokens (128 rows)
    check_block(block_inputs(B=32, n=4, seed=95))
