"""kda_block_tkg on the GPU (through the C ABI) against the float64 oracle.

Every buffer the block writes -- out, S, conv_state and its workspace -- is
guarded on both sides and checked after each call."""
import numpy as np
import pytest
import torch

import oracle
from kda_decode_recurrence_gb300 import _lib, block_workspace_size, kda_block_tkg, tp
from kda_decode_recurrence_gb300.inputs import block_inputs, to_f64

from _parity import (STATE_RTOL, Guarded, assert_outputs_close, assert_states_close,
                     guarded_copy, to_device)

pytestmark = pytest.mark.gpu

WEIGHTS = ("hidden", "gamma_in", "W_in", "W_fb", "W_gb", "conv_w", "A_log", "dt_bias",
           "gamma_o", "W_o")


def gpu_block(inp, workspace=None):
    d = to_device(inp)
    out = Guarded((inp["B"], inp["n"], inp["Hd"]), torch.float32, fill=float("nan"))
    S, cs = guarded_copy(inp["S"]), guarded_copy(inp["conv_state"])
    ws = None
    if workspace is None:
        ws = Guarded((block_workspace_size(inp["B"], inp["n"], inp["Hd"], inp["nh"], inp["K"],
                                           inp["V"], inp["Kc"]),), torch.uint8, fill=0x3C)
        workspace = ws.t
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_block_tkg(out.t, *[d[k] for k in WEIGHTS], S.t, cs.t, inp["scale"],
                  inp["lower_bound"], inp["rms_norm_eps"], inp["l2_eps"], workspace=workspace,
                  dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for g, name in ((out, "out"), (S, "S"), (cs, "conv_state"), (ws, "workspace")):
        assert g is None or g.intact(), f"write outside {name}"
    return out.t, S.t, cs.t


def oracle_block(inp):
    return oracle.kda_block_tkg(*[to_f64(inp[k]) for k in WEIGHTS], to_f64(inp["S"]),
                                to_f64(inp["conv_state"]), inp["scale"], inp["lower_bound"],
                                inp["rms_norm_eps"], inp["l2_eps"])


def check_block(inp, ref=None):
    out, S, cs = gpu_block(inp)
    ref_out, ref_S, ref_cs = oracle_block(inp) if ref is None else ref
    assert_outputs_close(out.cpu().numpy(), ref_out, "out")
    # The same 1e-5 bound for any number of tokens: the forget gate amplifies
    # the error of its latent f_a up to |lower_bound| exp(A_log) / 4 = 20
    # times, so the projection computes the f_a (and g_a, beta) columns from
    # the activations at fp32 precision.
    assert_states_close(S.cpu().numpy(), ref_S, "S", tol=STATE_RTOL)
    # conv_state: the last Kc-1 pre-convolution inputs.  With one token the
    # older entries are exact copies shifted by one; entries that come from
    # this call's projection carry the GEMM's rounding.
    cs = cs.cpu().numpy()
    assert_outputs_close(cs, ref_cs, "conv_state")
    if inp["n"] == 1:
        np.testing.assert_array_equal(cs[..., :-1], to_f64(inp["conv_state"])[..., 1:])


def test_block_full_config(kimi_k3_block):
    inp, ref = kimi_k3_block
    check_block(inp, ref)


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


def test_swish_output_gate_variant_library():
    # The library built with the block's output gate as swish (z * sigmoid(z))
    # against the oracle's swish setting; everything else is the same chain.
    lib = _lib.load_variant("outgate_swish")
    for sizes in ({"B": 6, "Hd": 256, "nh": 8, "seed": 97}, {"B": 3, "n": 3, "Hd": 384, "nh": 16, "seed": 98}):
        inp = block_inputs(**sizes)
        d = to_device(inp)
        out = Guarded((inp["B"], inp["n"], inp["Hd"]), torch.float32, fill=float("nan"))
        S, cs = guarded_copy(inp["S"]), guarded_copy(inp["conv_state"])
        ws = Guarded((block_workspace_size(inp["B"], inp["n"], inp["Hd"], inp["nh"], inp["K"],
                                           inp["V"], inp["Kc"]),), torch.uint8, fill=0)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = lib.kda_block_tkg(
            out.t.data_ptr(), *[d[k].data_ptr() for k in WEIGHTS], S.t.data_ptr(), cs.t.data_ptr(),
            inp["scale"], inp["lower_bound"], inp["rms_norm_eps"], inp["l2_eps"], inp["B"], inp["n"],
            inp["Hd"], inp["nh"], inp["K"], inp["V"], inp["Kc"], ws.t.data_ptr(), ws.t.numel(),
            status.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert rc == 0 and status.item() == 0
        assert out.intact() and S.intact() and cs.intact() and ws.intact()
        ref_out, ref_S, ref_cs = oracle.kda_block_tkg(
            *[to_f64(inp[k]) for k in WEIGHTS], to_f64(inp["S"]), to_f64(inp["conv_state"]),
            inp["scale"], inp["lower_bound"], inp["rms_norm_eps"], inp["l2_eps"], out_gate="swish")
        assert_outputs_close(out.t.cpu().numpy(), ref_out, "out")
        assert_states_close(S.t.cpu().numpy(), ref_S, "S")
        assert_outputs_close(cs.t.cpu().numpy(), ref_cs, "conv_state")
        # and it is not the sigmoid block
        sig_out, _, _ = oracle_block(inp)
        assert np.abs(sig_out - ref_out).max() > 1e-2


@pytest.fixture(scope="module")
def kimi_k3_block():
    inp = block_inputs()
    return inp, oracle_block(inp)


@pytest.mark.parametrize("tp_size", [2, 4])
def test_tensor_parallel_shards_sum_to_the_whole_block(kimi_k3_block, tp_size):
    # The Kimi K3 block (B = 32, Hd = 4096, 32 heads) cut into tp_size head
    # shards (16 or 8 heads each), each run as its own kda_block_tkg call on
    # this GPU, as the ranks of a tensor-parallel group would; the sum of
    # their partial outs -- what the group's all-reduce produces -- is the
    # whole block's out, and the shards' states gather into its state.
    inp, (ref_out, ref_S, ref_cs) = kimi_k3_block
    d = to_device(inp)
    params = {k: d[k] for k in tp.BLOCK_PARAMS}
    total = torch.zeros((inp["B"], inp["n"], inp["Hd"]), dtype=torch.float64, device="cuda")
    S_parts, cs_parts = [], []
    for r in range(tp_size):
        shard = tp.shard_block_params(params, tp_size, r)
        S_r, cs_r = tp.shard_block_state(d["S"], d["conv_state"], tp_size, r)
        S_g, cs_g = guarded_copy(S_r), guarded_copy(cs_r)
        out = Guarded((inp["B"], inp["n"], inp["Hd"]), torch.float32, fill=float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda_block_tkg(out.t, d["hidden"], *[shard[k] for k in tp.BLOCK_PARAMS], S_g.t, cs_g.t,
                      inp["scale"], inp["lower_bound"], inp["rms_norm_eps"], inp["l2_eps"],
                      dev_status=status)
        torch.cuda.synchronize()
        assert status.item() == 0 and out.intact() and S_g.intact() and cs_g.intact()
        total += out.t.double()
        S_parts.append(S_g.t)
        cs_parts.append(cs_g.t)
    S_all, cs_all = tp.gather_block_state(S_parts, cs_parts)
    assert_outputs_close(total.cpu().numpy(), ref_out, "sum of partial outs")
    assert_states_close(S_all.cpu().numpy(), ref_S, "S")
    assert_outputs_close(cs_all.cpu().numpy(), ref_cs, "conv_state")
