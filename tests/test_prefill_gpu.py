"""kda_prefill (the chunked whole-sequence form) on the GPU against the
float64 oracle, and against kda_decode's token-by-token kernel on a full-size
prompt."""
import numpy as np
import pytest
import torch

from kda_decode_recurrence_gb300 import DEV_BAD_SLOT, kda_decode, kda_prefill
from kda_decode_recurrence_gb300.inputs import decode_inputs

from _parity import (Guarded, assert_outputs_close, assert_states_close, guarded_copy,
                     oracle_decode_sample, to_device)

pytestmark = pytest.mark.gpu


def gpu_prefill(inp, fn=kda_prefill):
    d = to_device(inp)
    out = Guarded((inp["T"], inp["HV"], inp["V"]), torch.float32, fill=float("nan"))
    pool = guarded_copy(inp["state_pool"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn(out.t, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"], d["dt_bias"],
       d["cu_seqlens"], pool.t, d["state_indices"], gate_mode=inp["gate_mode"],
       lower_bound=inp["lower_bound"], dev_status=status)
    torch.cuda.synchronize()
    assert out.intact() and pool.intact()
    return out.t, pool.t, int(status.item())


def check(inp, bs=None, state_tol=1e-5):
    out, pool, st = gpu_prefill(inp)
    assert st == 0
    bs = list(range(inp["B"])) if bs is None else bs
    rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, bs)
    assert_outputs_close(out.cpu().numpy()[rows], ref_out)
    assert_states_close(pool[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy(),
                        ref_pool, tol=state_tol)


@pytest.mark.parametrize("lb", [-5.0, -1.0, 0.0])
def test_chunk_boundaries_against_oracle(lb):
    # lb = 0: every g is 0, no decay at all (the degenerate end of the gate)
    # partial chunks, exactly one chunk, one past a chunk, several chunks
    inp = decode_inputs("varlen", B=6, H=2, HV=4, max_slots=8,
                        lengths=(1, 15, 16, 17, 40, 100), seed=120)
    inp["lower_bound"] = lb
    check(inp)


def test_many_ragged_requests_with_empty_ones():
    # one launch over requests of very different chunk counts, some of them
    # empty: every request and head against the oracle, the empty requests'
    # tiles bit-identical
    rng = np.random.default_rng(126)
    lengths = [int(x) for x in rng.integers(0, 150, size=24)]
    lengths[3] = lengths[11] = lengths[20] = 0
    inp = decode_inputs("varlen", B=24, H=4, HV=8, max_slots=30, lengths=tuple(lengths), seed=126)
    out, pool, st = gpu_prefill(inp)
    assert st == 0
    idx = inp["state_indices"].numpy()
    for b in (3, 11, 20):
        assert torch.equal(pool[int(idx[b])].cpu(), inp["state_pool"][int(idx[b])])
    rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, list(range(24)))
    assert_outputs_close(out.cpu().numpy()[rows], ref_out)
    assert_states_close(pool[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy(), ref_pool)


def test_long_sequence_against_oracle():
    inp = decode_inputs("varlen", B=2, H=4, HV=4, max_slots=3, lengths=(1000, 777), seed=121)
    check(inp)


def test_grouped_heads_against_oracle():
    inp = decode_inputs("varlen", B=3, H=2, HV=8, max_slots=5, lengths=(33, 64, 5), seed=122)
    check(inp)


def test_matches_token_by_token_kernel_on_a_full_prompt():
    # the bench's prefill workload: 2 requests x 2048 tokens, 96 heads
    inp = decode_inputs("varlen", B=2, H=96, HV=96, max_slots=4, lengths=(2048, 2048), seed=7)
    out_c, pool_c, st_c = gpu_prefill(inp)
    out_r, pool_r, st_r = gpu_prefill(inp, fn=kda_decode)
    assert st_c == 0 and st_r == 0
    assert_outputs_close(out_c.cpu().numpy(), out_r.cpu().double().numpy(), "out")
    slots = inp["state_indices"].long().cuda()
    assert_states_close(pool_c[slots].cpu().numpy(), pool_r[slots].cpu().double().numpy(), "S")
    # and a sample of it against the oracle
    rows, sl, ref_out, ref_pool = oracle_decode_sample(
        {**inp, "HV": 96}, [0])
    assert_outputs_close(out_c.cpu().numpy()[rows], ref_out)


def test_padded_and_out_of_range_slots():
    inp = decode_inputs("varlen", B=4, H=2, HV=2, max_slots=5, lengths=(20, 3, 17, 2), seed=123)
    inp["state_indices"] = torch.tensor([2, -1, 4, 9], dtype=torch.int32)
    out, pool, st = gpu_prefill(inp)
    assert st == DEV_BAD_SLOT
    cu = inp["cu_seqlens"].numpy()
    o = out.cpu().numpy()
    assert np.all(o[cu[1]:cu[2]] == 0.0) and np.all(o[cu[3]:cu[4]] == 0.0)
    for s in (0, 1, 3):
        assert torch.equal(pool[s].cpu(), inp["state_pool"][s])
    rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, [0, 2])
    assert_outputs_close(o[rows], ref_out)
    assert_states_close(pool[torch.tensor(slots.astype(np.int64)).cuda()].cpu().numpy(), ref_pool)


def test_q_k_v_at_an_8_byte_offset():
    # The C ABI asks for 8-byte alignment of q, k, v; the chunk copies use
    # 16-byte pieces only when all three are 16-byte aligned.  Views at an
    # 8-byte offset take the 8-byte path and must give the same results.
    inp = decode_inputs("varlen", B=3, H=2, HV=4, max_slots=5, lengths=(37, 16, 70), seed=124)
    d = to_device(inp)
    views = {}
    for name in ("q", "k", "v"):
        t = d[name]
        buf = torch.empty(t.numel() + 4, dtype=t.dtype, device="cuda")
        view = buf[4:].view(t.shape)
        view.copy_(t)
        assert view.data_ptr() % 16 == 8
        views[name] = view
    out_a, pool_a, st_a = gpu_prefill(inp)
    out = torch.full_like(out_a, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_prefill(out, views["q"], views["k"], views["v"], d["raw_gate"], d["beta_logits"],
                d["a_log"], d["dt_bias"], d["cu_seqlens"], d["state_pool"], d["state_indices"],
                gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"], dev_status=status)
    torch.cuda.synchronize()
    assert st_a == 0 and int(status.item()) == 0
    # same arithmetic in the same order: bit-identical
    assert torch.equal(out, out_a)
    slots = inp["state_indices"].long().cuda()
    assert torch.equal(d["state_pool"][slots], pool_a[slots])


@pytest.mark.parametrize("gate,lb", [(0, -5.0), (1, -6.0)])
def test_gates_outside_the_chunk_form_run_the_token_kernel(gate, lb):
    # the softplus gate (unbounded decay) and lower bounds below -5 cannot use
    # the chunk form: kda_prefill then runs the token-by-token kernel, so its
    # results are kda_decode's bit for bit, and the oracle's within the bounds
    inp = decode_inputs("varlen", B=4, H=2, HV=4, max_slots=6, lengths=(40, 1, 17, 33), seed=125)
    inp["gate_mode"], inp["lower_bound"] = gate, lb
    out_p, pool_p, st_p = gpu_prefill(inp)
    out_d, pool_d, st_d = gpu_prefill(inp, fn=kda_decode)
    assert st_p == 0 and st_d == 0
    assert torch.equal(out_p, out_d) and torch.equal(pool_p, pool_d)
    check(inp)


def test_many_waves_of_ctas_match_the_token_kernel():
    # 64 requests x 96 heads = 6144 CTAs, about 20 waves at two per SM: every
    # wave allocates and frees its tensor memory; the results equal the
    # token-by-token kernel's within the bounds, and a sample the oracle's
    inp = decode_inputs("varlen", B=64, H=96, HV=96, max_slots=128, seed=128,
                        lengths=tuple(int(x) for x in np.random.default_rng(128).integers(1, 100, 64)))
    out_c, pool_c, st_c = gpu_prefill(inp)
    out_r, pool_r, st_r = gpu_prefill(inp, fn=kda_decode)
    assert st_c == 0 and st_r == 0
    assert_outputs_close(out_c.cpu().numpy(), out_r.cpu().double().numpy(), "out")
    slots = inp["state_indices"].long().cuda()
    assert_states_close(pool_c[slots].cpu().numpy(), pool_r[slots].cpu().double().numpy(), "S")
    rows, sl, ref_out, ref_pool = oracle_decode_sample(inp, [0, 31, 63])
    assert_outputs_close(out_c.cpu().numpy()[rows], ref_out)
    assert_states_close(pool_c[torch.from_numpy(sl.astype(np.int64)).cuda()].cpu().numpy(), ref_pool)


def test_prefill_then_decode_steps_equal_one_pass():
    # the serving flow: a prompt prefilled in chunks, then tokens decoded one
    # call each on the same pool, against the oracle over all the tokens
    P, steps = 70, 3
    inp = decode_inputs("varlen", B=3, H=2, HV=4, max_slots=5, lengths=(P + steps,) * 3, seed=127)
    d = to_device(inp)
    B, HV = inp["B"], inp["HV"]
    T = P + steps
    tok = {k: d[k].view(B, T, *d[k].shape[1:]) for k in ("q", "k", "v", "raw_gate", "beta_logits")}
    pool = d["state_pool"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((B, T, HV, 128), float("nan"), device="cuda")
    seg = lambda name, a, b: tok[name][:, a:b].reshape(-1, *tok[name].shape[2:]).contiguous()
    cu = lambda n: torch.arange(0, B * n + 1, n, dtype=torch.int32, device="cuda")
    o = torch.empty(B * P, HV, 128, device="cuda")
    kda_prefill(o, seg("q", 0, P), seg("k", 0, P), seg("v", 0, P), seg("raw_gate", 0, P),
                seg("beta_logits", 0, P), d["a_log"], d["dt_bias"], cu(P), pool, d["state_indices"],
                gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"], dev_status=status)
    out[:, :P] = o.view(B, P, HV, 128)
    for j in range(P, T):
        o1 = torch.empty(B, HV, 128, device="cuda")
        kda_decode(o1, seg("q", j, j + 1), seg("k", j, j + 1), seg("v", j, j + 1),
                   seg("raw_gate", j, j + 1), seg("beta_logits", j, j + 1), d["a_log"], d["dt_bias"],
                   cu(1), pool, d["state_indices"], gate_mode=inp["gate_mode"],
                   lower_bound=inp["lower_bound"], dev_status=status)
        out[:, j] = o1
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, list(range(B)))
    assert_outputs_close(out.view(B * T, HV, 128).cpu().numpy()[rows], ref_out)
    assert_states_close(pool[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy(), ref_pool)
