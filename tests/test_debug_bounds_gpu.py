"""The debug build's index checks (libkda_debugbounds.so, KDA_DEBUG_BOUNDS=1).

That build adds a check to the kernels' derived indices (request, heads,
slot, token rows, output rows, block rows) before the global accesses they
guard: a failed check sets KDA_DEV_BOUNDS in the status word and skips the
access instead of performing it.  It is the stand-in for a bounds-checking
tool.  On valid inputs no check may fire, and the checks must not change any
result: each call below runs through both libraries on the same inputs and
must give status 0 and bit-identical outputs and states (the block within
rounding, see below).
"""
import pytest
import torch

from kda_decode_recurrence_gb300 import _lib
from kda_decode_recurrence_gb300.inputs import block_inputs, decode_inputs

from _parity import to_device

pytestmark = pytest.mark.gpu

BLOCK_W = ("hidden", "gamma_in", "W_in", "W_fb", "W_gb", "conv_w", "A_log", "dt_bias",
           "gamma_o", "W_o")


def libs():
    return {"product": _lib.load(), "debug": _lib.load_variant("debugbounds")}


def run_decode(lib, inp, fn="kda_decode", state_layout=0, output_dtype=0):
    d = to_device(inp)
    pool = d["state_pool"].clone()
    if state_layout == 1:
        pool = pool.transpose(-1, -2).contiguous()
    dtype = torch.float32 if output_dtype == 0 else torch.bfloat16
    out = torch.full((inp["T"], inp["HV"], 128), float("nan"), dtype=dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = [out.data_ptr(), d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
            d["raw_gate"].data_ptr(), d["beta_logits"].data_ptr(), d["a_log"].data_ptr(),
            d["dt_bias"].data_ptr(), d["cu_seqlens"].data_ptr(), pool.data_ptr(),
            d["state_indices"].data_ptr(), inp["gate_mode"], inp["lower_bound"]]
    if fn == "kda_decode_ex":
        args += [state_layout, output_dtype]
    args += [inp["B"], inp["T"], inp["H"], inp["HV"], 128, 128, inp["max_slots"],
             status.data_ptr(), torch.cuda.current_stream().cuda_stream]
    assert getattr(lib, fn)(*args) == 0
    torch.cuda.synchronize()
    return out, pool, int(status.item())


def run_block(lib, b, n):
    d = to_device(b)
    S, conv = d["S"].clone(), d["conv_state"].clone()
    B, Hd, nh, Kc = b["B"], b["Hd"], b["nh"], b["Kc"]
    out = torch.full((B, n, Hd), float("nan"), device="cuda")
    ws = torch.empty(lib.kda_block_tkg_workspace_size(B, n, Hd, nh, 128, 128, Kc),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.kda_block_tkg(out.data_ptr(), *[d[k].data_ptr() for k in BLOCK_W], S.data_ptr(),
                             conv.data_ptr(), b["scale"], b["lower_bound"], b["rms_norm_eps"],
                             b["l2_eps"], B, n, Hd, nh, 128, 128, Kc, ws.data_ptr(), ws.numel(),
                             status.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    return out, S, conv, int(status.item())


def same(results):
    prod, dbg = results["product"], results["debug"]
    assert dbg[-1] == 0, f"debug build status {dbg[-1]}"
    assert prod[-1] == 0
    for a, b in zip(prod[:-1], dbg[:-1]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("wl,kw", [
    ("grouped", dict(B=32, max_slots=64)),                    # single-token kernel, G = 2
    ("varlen", dict(B=24, H=8, HV=16, max_slots=32)),         # multi-token kernel, balanced order
    ("varlen", dict(B=4, H=2, HV=4, max_slots=8, lengths=(0, 9, 17, 3))),
])
def test_decode_checks_silent_and_results_unchanged(wl, kw):
    inp = decode_inputs(wl, **kw)
    same({name: run_decode(lib, inp) for name, lib in libs().items()})


def test_decode_v_first_bf16_checks_silent():
    inp = decode_inputs("varlen", B=8, H=4, HV=8, max_slots=12)
    same({name: run_decode(lib, inp, "kda_decode_ex", 1, 1) for name, lib in libs().items()})


def test_prefill_checks_silent_and_results_unchanged():
    inp = decode_inputs("varlen", B=5, H=2, HV=4, max_slots=8, lengths=(1, 16, 40, 0, 33))
    same({name: run_decode(lib, inp, "kda_prefill") for name, lib in libs().items()})


@pytest.mark.parametrize("n", [1, 4])
def test_block_checks_silent_and_results_unchanged(n):
    # The block's projections add their split-K partial sums with fp32
    # atomics (the g_a, beta, f_a columns and out), whose order varies from
    # call to call, so out and S are compared within rounding; conv_state
    # (the projection's q, k, v columns, summed in a fixed order) exactly.
    b = block_inputs(B=3, Hd=256, nh=8, n=n, seed=30 + n)
    r = {name: run_block(lib, b, n) for name, lib in libs().items()}
    (out_p, S_p, conv_p, st_p), (out_d, S_d, conv_d, st_d) = r["product"], r["debug"]
    assert st_p == 0 and st_d == 0, (st_p, st_d)
    assert torch.equal(conv_p, conv_d)
    assert torch.allclose(out_d, out_p, rtol=1e-5, atol=1e-6)
    assert torch.allclose(S_d, S_p, rtol=1e-5, atol=1e-7)
