"""kda_decode on the GPU (through the C ABI) against the float64 oracle.

Full-size workloads (single, grouped, varlen) run in the launch configuration
the benchmark times; the oracle then checks every request (all token rows,
all advanced tiles), and the untouched part of the pool is compared bit for
bit.  Small and ragged cases are compared in full.  Every buffer a kernel
writes is guarded on both sides (tests/_parity.py, Guarded).
"""
import numpy as np
import pytest
import torch

import oracle

from kda_decode_recurrence_gb300 import DEV_BAD_SEQLEN, DEV_BAD_SLOT, GATE_LOWER_BOUND, kda_decode
from kda_decode_recurrence_gb300.inputs import decode_inputs, to_f64

from _parity import (Guarded, assert_all_requests_match, assert_outputs_close,
                     assert_states_close, gpu_decode, guarded_copy, oracle_decode_sample,
                     to_device)

pytestmark = pytest.mark.gpu


def check_all(inp, bs=None):
    out, pool, st = gpu_decode(inp)
    assert st == 0
    B = inp["B"]
    bs = list(range(B)) if bs is None else bs
    rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, bs)
    assert_outputs_close(out.cpu().numpy()[rows], ref_out)
    assert_states_close(pool[torch.from_numpy(slots.astype(np.int64))].cpu().numpy(), ref_pool)
    return out, pool


def test_tiny_full():
    check_all(decode_inputs("tiny"))


@pytest.mark.parametrize("name", ["single", "grouped", "varlen"])
def test_full_size_every_request(name):
    inp = decode_inputs(name)
    d = to_device(inp)
    pool = guarded_copy(inp["state_pool"])
    before = pool.t.clone()
    out = Guarded((inp["T"], inp["HV"], inp["V"]), torch.float32, fill=float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_decode(out.t, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
               d["dt_bias"], d["cu_seqlens"], pool.t, d["state_indices"],
               gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"], dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert out.intact() and pool.intact()
    assert torch.isfinite(out.t).all().item()          # every token row written
    # every request: all of its token rows and all HV of its advanced tiles
    assert assert_all_requests_match(inp, out.t, pool.t) == inp["B"]
    used = torch.zeros(inp["max_slots"], dtype=torch.bool, device="cuda")
    used[d["state_indices"].long()] = True
    assert torch.equal(pool.t[~used], before[~used])   # untouched slots bit-identical


@pytest.mark.parametrize("gate", [0, 1])
@pytest.mark.parametrize("H,HV", [(3, 6), (2, 2), (1, 4)])
def test_ragged_varlen_small(gate, H, HV):
    # lengths include an empty request, one token, more than one staging round
    # (> 8 tokens) and a ragged last round
    lengths = (0, 1, 9, 17, 3)
    inp = decode_inputs("varlen", B=5, H=H, HV=HV, max_slots=11, lengths=lengths, seed=40 + gate)
    inp["gate_mode"] = gate
    out, pool = check_all(inp, bs=[1, 2, 3, 4])
    empty_slot = int(inp["state_indices"][0])
    assert torch.equal(pool[empty_slot].cpu(), inp["state_pool"][empty_slot])


def test_padded_and_out_of_range_slots():
    inp = decode_inputs("varlen", B=4, H=2, HV=4, max_slots=6, lengths=(2, 1, 3, 2), seed=50)
    inp["state_indices"] = torch.tensor([3, -1, 1, 6], dtype=torch.int32)  # 6 == max_slots: bad
    out, pool, st = gpu_decode(inp)
    assert st == DEV_BAD_SLOT
    cu = inp["cu_seqlens"].numpy()
    o = out.cpu().numpy()
    assert np.all(o[cu[1]:cu[2]] == 0.0) and np.all(o[cu[3]:cu[4]] == 0.0)
    for s in (0, 2, 4, 5):
        assert torch.equal(pool[s].cpu(), inp["state_pool"][s])
    rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, [0, 2])
    assert_outputs_close(o[rows], ref_out)
    assert_states_close(pool[torch.tensor(slots.astype(np.int64))].cpu().numpy(), ref_pool)


@pytest.mark.parametrize("cu", [[0, 3, 2, 6], [0, 2, 4, 7], [1, 2, 4, 6]])
def test_malformed_cu_seqlens_flagged(cu):
    inp = decode_inputs("varlen", B=3, H=2, HV=2, max_slots=4, lengths=(2, 2, 2), seed=51)
    inp["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    out, pool, st = gpu_decode(inp, output_fill=0.0)
    assert st & DEV_BAD_SEQLEN


def test_no_tokens_is_a_no_op():
    inp = decode_inputs("varlen", B=3, H=2, HV=2, max_slots=4, lengths=(0, 0, 0), seed=52)
    d = to_device(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(0, 2, 128, device="cuda")
    kda_decode(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
               d["dt_bias"], d["cu_seqlens"], d["state_pool"], d["state_indices"],
               dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(d["state_pool"].cpu(), inp["state_pool"])


def test_multi_token_call_equals_single_token_calls():
    inp = decode_inputs("varlen", B=4, H=2, HV=4, max_slots=5, lengths=(5, 1, 12, 3), seed=53)
    out_all, pool_all, st = gpu_decode(inp)
    assert st == 0
    d = to_device(inp)
    cu = inp["cu_seqlens"].tolist()
    out_step = torch.empty_like(out_all)
    for b in range(4):
        for t in range(cu[b], cu[b + 1]):
            o = torch.empty(1, 4, 128, device="cuda")
            kda_decode(o, d["q"][t:t + 1], d["k"][t:t + 1], d["v"][t:t + 1],
                       d["raw_gate"][t:t + 1], d["beta_logits"][t:t + 1], d["a_log"], d["dt_bias"],
                       torch.tensor([0, 1], dtype=torch.int32, device="cuda"), d["state_pool"],
                       d["state_indices"][b:b + 1].contiguous(), gate_mode=inp["gate_mode"],
                       lower_bound=inp["lower_bound"])
            out_step[t] = o[0]
    torch.cuda.synchronize()
    # the tile is stored in fp32 exactly as held on chip, so chaining calls is
    # bit-identical to one call
    assert torch.equal(out_step, out_all)
    assert torch.equal(d["state_pool"], pool_all)


def test_same_token_read_returns_value_at_full_size():
    # beta = 1 and q = k: q^T S_new = K^-1/2 v for any state and gate (the
    # delta-rule property), up to the l2_eps term (~1e-8 relative here).
    # Element by element: the l2_eps term moves o by about 1e-8 |v| and the
    # fp32 arithmetic by a few 1e-8 |v|, well inside 1e-6 (1 + |v|).
    inp = decode_inputs("grouped")
    inp["q"] = inp["k"].clone()
    inp["beta_logits"] = torch.full_like(inp["beta_logits"], 40.0)
    out, _, st = gpu_decode(inp)
    assert st == 0
    v = to_f64(inp["v"])
    err = np.abs(out.cpu().numpy() - v * 128 ** -0.5)
    assert np.all(err <= 1e-6 * (1 + np.abs(v))), float((err / (1 + np.abs(v))).max())


def test_lower_bound_gate_never_amplifies_on_gpu():
    inp = decode_inputs("varlen", B=8, H=4, HV=4, max_slots=8, lengths=(1,) * 8, seed=54)
    inp["gate_mode"] = GATE_LOWER_BOUND
    inp["beta_logits"] = torch.full_like(inp["beta_logits"], -200.0)   # beta == 0: decay only
    inp["raw_gate"] = inp["raw_gate"] * 10
    _, pool, st = gpu_decode(inp)
    assert st == 0
    slots = inp["state_indices"].long()
    ratio = (pool[slots.cuda()].cpu() / inp["state_pool"][slots]).numpy()
    assert np.all(ratio <= 1.0) and np.all(ratio >= np.exp(-5.0) * (1 - 1e-6))


def test_beta_zero_scales_each_state_row_and_nothing_else():
    # beta == 0 (sigmoid(-200) is 0 in fp32): the step is the decay alone, so
    # every row k of the advanced tile is the old row times one factor exp(g_k)
    # (one fp32 rounding per element), and that factor is the oracle's.
    inp = decode_inputs("varlen", B=6, H=2, HV=4, max_slots=8, lengths=(1,) * 6, seed=55)
    inp["beta_logits"] = torch.full_like(inp["beta_logits"], -200.0)
    out, pool, st = gpu_decode(inp)
    assert st == 0
    slots = inp["state_indices"].long()
    before = to_f64(inp["state_pool"][slots])
    after = pool[slots.cuda()].cpu().double().numpy()
    ratio = after / before                                   # [B, HV, K, V]
    row = np.median(ratio, axis=-1, keepdims=True)
    assert np.all(np.abs(ratio - row) <= 2.0 ** -22 * np.abs(row))
    rows, _, ref_out, ref_pool = oracle_decode_sample(inp, range(inp["B"]))
    ref_ratio = ref_pool[..., :1] / before[..., :1]
    np.testing.assert_allclose(row, ref_ratio, rtol=1e-4)
    assert_outputs_close(out.cpu().numpy()[rows], ref_out)


def test_grouped_heads_equal_duplicated_heads_bit_for_bit():
    # G = 2 (H = 48 key heads for HV = 96 value heads) is the same computation
    # as H = 96 with each key head's q and k repeated for its two value heads.
    inp = decode_inputs("grouped")
    out_g, pool_g, st_g = gpu_decode(inp)
    dup = dict(inp)
    dup["q"] = inp["q"].repeat_interleave(2, dim=1).contiguous()
    dup["k"] = inp["k"].repeat_interleave(2, dim=1).contiguous()
    out_d, pool_d, st_d = gpu_decode(dup)
    assert st_g == 0 and st_d == 0
    assert torch.equal(out_g, out_d)
    assert torch.equal(pool_g, pool_d)


def test_permuting_requests_with_their_slots_permutes_the_outputs():
    lengths = (3, 1, 5, 2, 4, 1, 9)
    inp = decode_inputs("varlen", B=7, H=2, HV=4, max_slots=10, lengths=lengths, seed=56)
    out, pool, st = gpu_decode(inp)
    assert st == 0
    perm = [4, 0, 6, 2, 5, 1, 3]
    cu = inp["cu_seqlens"].tolist()
    rows = torch.cat([torch.arange(cu[b], cu[b + 1]) for b in perm])
    new_len = [lengths[b] for b in perm]
    moved = dict(inp)
    for key in ("q", "k", "v", "raw_gate", "beta_logits"):
        moved[key] = inp[key][rows].contiguous()
    moved["cu_seqlens"] = torch.tensor(np.concatenate([[0], np.cumsum(new_len)]), dtype=torch.int32)
    moved["state_indices"] = inp["state_indices"][perm].contiguous()
    out_p, pool_p, st_p = gpu_decode(moved)
    assert st_p == 0
    assert torch.equal(out_p, out[rows.cuda()])
    assert torch.equal(pool_p, pool)


def test_persistent_ring_with_mixed_items():  # noqa: C901
    # Many more (request, head) items than SMs, so every CTA cycles through its
    # copy ring many times, with padded, out-of-range and empty requests mixed
    # in (their ring slots are consumed without a tile).
    rng = np.random.default_rng(77)
    B, HV, N = 400, 2, 430
    lengths = rng.integers(0, 4, size=B)
    inp = decode_inputs("varlen", B=B, H=1, HV=HV, max_slots=N, lengths=lengths, seed=78)
    idx = inp["state_indices"].numpy().copy()
    padded = rng.choice(B, size=30, replace=False)
    idx[padded[:20]] = -1
    idx[padded[20:]] = N + 5                      # out of range
    inp["state_indices"] = torch.from_numpy(idx)
    d = to_device(inp)
    pool = guarded_copy(inp["state_pool"])
    d["state_pool"] = pool.t
    before = pool.t.clone()
    gout = Guarded((inp["T"], HV, 128), torch.float32, fill=float("nan"))
    out = gout.t
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_decode(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
               d["dt_bias"], d["cu_seqlens"], d["state_pool"], d["state_indices"],
               gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"], dev_status=status)
    torch.cuda.synchronize()
    assert gout.intact() and pool.intact()
    assert status.item() == DEV_BAD_SLOT
    cu = inp["cu_seqlens"].numpy()
    o = out.cpu().numpy()
    for b in padded:
        assert np.all(o[cu[b]:cu[b + 1]] == 0.0)
    valid = [b for b in range(B) if idx[b] >= 0 and idx[b] < N]
    rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, valid)
    assert_outputs_close(o[rows], ref_out)
    assert_states_close(d["state_pool"][torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy(),
                        ref_pool)
    advanced = set(int(idx[b]) for b in valid if lengths[b] > 0)
    untouched = torch.tensor([s for s in range(N) if s not in advanced], device="cuda")
    assert torch.equal(d["state_pool"][untouched], before[untouched])


# ------------------------------------------------ kda_decode_ex (layout, dtype)

from kda_decode_recurrence_gb300 import STATE_V_FIRST, kda_decode_ex  # noqa: E402


def run_ex(inp, v_first, out_dtype, dev="cuda"):
    d = to_device(inp, dev)
    src = inp["state_pool"].transpose(-1, -2).contiguous() if v_first else inp["state_pool"]
    gpool = guarded_copy(src, dev)
    pool = gpool.t
    gout = Guarded((inp["T"], inp["HV"], inp["V"]), out_dtype, dev, fill=float("nan"))
    out = gout.t
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kda_decode_ex(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
                  d["dt_bias"], d["cu_seqlens"], pool, d["state_indices"],
                  gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"],
                  state_layout=STATE_V_FIRST if v_first else 0, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert gout.intact() and gpool.intact()
    kfirst = pool.transpose(-1, -2) if v_first else pool
    return out, kfirst


@pytest.mark.parametrize("gate", [0, 1])
@pytest.mark.parametrize("name", ["tiny", "varlen_small"])
def test_v_first_and_bf16_output_against_oracle(name, gate):
    # The transposed tiles are held by the lanes as runs of 4 rows, so their
    # k-contractions add the rows in another order than the row-major form:
    # both are checked against the oracle, and against each other within the
    # same bounds.  The bf16 output is the same computation rounded at the
    # store: exactly the fp32 output rounded to nearest even, with the same
    # advanced pool bit for bit.
    inp = (decode_inputs("tiny") if name == "tiny" else
           decode_inputs("varlen", B=6, H=2, HV=4, max_slots=9, lengths=(1, 0, 9, 3, 17, 2), seed=90))
    inp["gate_mode"] = gate
    vf_out, vf_pool = run_ex(inp, True, torch.float32)
    bs = [b for b in range(inp["B"]) if int(inp["state_indices"][b]) >= 0]
    rows, slots, ref_out, ref_pool = oracle_decode_sample(inp, bs)
    assert_outputs_close(vf_out.cpu().numpy()[rows], ref_out)
    assert_states_close(vf_pool[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy(),
                        ref_pool)
    kf_out, kf_pool = run_ex(inp, False, torch.float32)
    assert_outputs_close(kf_out.cpu().numpy()[rows], vf_out.cpu().double().numpy()[rows])
    assert_states_close(kf_pool.cpu().numpy(), vf_pool.cpu().double().numpy())
    bf_out, bf_pool = run_ex(inp, True, torch.bfloat16)
    fin = torch.isfinite(vf_out)
    assert torch.equal(torch.isfinite(bf_out), fin)
    assert torch.equal(bf_out[fin], vf_out[fin].to(torch.bfloat16))   # round to nearest even
    assert torch.equal(bf_pool, vf_pool)


@pytest.mark.parametrize("name", ["grouped", "varlen"])
def test_v_first_bf16_full_size_against_oracle(name):
    # every request of the workload, V-first tiles, bf16 output (varlen: the
    # multi-token kernel)
    inp = decode_inputs(name)
    out, pool = run_ex(inp, True, torch.bfloat16)

    def bf16_bound(got, ref):
        # the fp32 bound plus one bf16 unit in the last place (2^-8 relative)
        err = np.abs(got - ref)
        assert np.all(err <= 1e-3 * (1 + np.abs(ref)) + 2.0 ** -8 * np.abs(ref))

    assert assert_all_requests_match(inp, out, pool, out_bound=bf16_bound) == inp["B"]


def test_pool_larger_than_4_gib():
    # 4096 slots x 96 heads x 64 KiB = 25.8 GB: tile byte offsets far beyond
    # 32 bits.  Only the touched slots (and neighbours used as sentinels) are
    # filled; the oracle runs on a compact pool holding the same tiles.
    small = decode_inputs("grouped", B=4, max_slots=4, seed=130)
    big_slot = torch.tensor([0, 1234, 4094, 4095])
    d = to_device(small)
    pool = torch.empty((4096, small["HV"], 128, 128), dtype=torch.float32, device="cuda")
    pool[big_slot.cuda()] = d["state_pool"]
    sentinels = torch.tensor([1, 1233, 1235, 4093]).cuda()
    pool[sentinels] = 7.0
    idx = big_slot[small["state_indices"].long()].to(torch.int32).cuda()
    out = torch.full((small["T"], small["HV"], small["V"]), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_decode(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
               d["dt_bias"], d["cu_seqlens"], pool, idx, gate_mode=small["gate_mode"],
               lower_bound=small["lower_bound"], dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    rows, slots, ref_out, ref_pool = oracle_decode_sample(small, range(small["B"]))
    assert_outputs_close(out[torch.from_numpy(rows).cuda()].cpu().numpy(), ref_out)
    got = pool[big_slot[torch.from_numpy(slots.astype(np.int64))].cuda()].cpu().numpy()
    assert_states_close(got, ref_pool)
    assert bool((pool[sentinels] == 7.0).all())
    del pool
    torch.cuda.empty_cache()


def test_multi_token_items_beyond_the_descriptor_table():
    # The multi-token kernel (T > B) keeps up to 512 item descriptors per CTA
    # in shared memory and reads any later ones from global memory.  With more
    # than 512 items per CTA (a persistent grid of 2 CTAs per SM), every CTA
    # crosses that boundary.  The pool then holds over 10 GB of tiles: only
    # the sampled requests' slots get seeded values, the rest stay zero (a
    # valid state); requests on both sides of the boundary are checked.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid = 2 * sms
    H = HV = 32
    B = (512 * grid) // HV + 40                      # 40 requests' items past the table
    lengths = 1 + np.arange(B) % 2                   # T > B: the multi-token kernel
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    rng = np.random.default_rng(150)
    tok = {"q": rng.standard_normal((T, H, 128), dtype=np.float32),
           "k": rng.standard_normal((T, H, 128), dtype=np.float32),
           "v": rng.standard_normal((T, HV, 128), dtype=np.float32),
           "raw_gate": rng.standard_normal((T, HV, 128), dtype=np.float32),
           "beta_logits": rng.standard_normal((T, HV), dtype=np.float32)}
    a_log = np.log(rng.uniform(1, 16, HV)).astype(np.float32)
    dt_bias = (0.1 * rng.standard_normal((HV, 128))).astype(np.float32)
    sample = list(range(8)) + list(range(B - 64, B))
    slots = rng.permutation(B).astype(np.int32)       # request b -> slot slots[b]
    tiles = (0.05 * rng.standard_normal((len(sample), HV, 128, 128))).astype(np.float32)
    dev = "cuda"
    tq = {k_: torch.from_numpy(v_) for k_, v_ in tok.items()}
    for name in ("q", "k", "v"):
        tq[name] = tq[name].to(torch.bfloat16)
    d = {k_: v_.to(dev) for k_, v_ in tq.items()}
    pool = Guarded((B, HV, 128, 128), torch.float32, dev, fill=0.0)
    pool.t[torch.from_numpy(slots[sample].astype(np.int64)).to(dev)] = torch.from_numpy(tiles).to(dev)
    out = Guarded((T, HV, 128), torch.float32, dev, fill=float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kda_decode(out.t, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"],
               torch.from_numpy(a_log).to(dev), torch.from_numpy(dt_bias).to(dev),
               torch.from_numpy(cu).to(dev), pool.t, torch.from_numpy(slots).to(dev),
               gate_mode=GATE_LOWER_BOUND, lower_bound=-5.0, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0 and out.intact() and pool.intact()
    assert torch.isfinite(out.t).all().item()
    # the oracle on the sampled requests, with their exact (bf16-rounded) inputs
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in sample])
    sub = {k_: to_f64(tq[k_][torch.from_numpy(rows)]) for k_ in tq}
    ref_out, ref_pool, st = oracle.kda_decode(
        sub["q"], sub["k"], sub["v"], sub["raw_gate"], sub["beta_logits"], a_log.astype(np.float64),
        dt_bias.astype(np.float64), np.concatenate([[0], np.cumsum(lengths[sample])]),
        tiles.astype(np.float64), np.arange(len(sample)), gate_mode=GATE_LOWER_BOUND,
        lower_bound=-5.0)
    assert st == 0
    assert_outputs_close(out.t[torch.from_numpy(rows).to(dev)].cpu().numpy(), ref_out)
    got = pool.t[torch.from_numpy(slots[sample].astype(np.int64)).to(dev)].cpu().numpy()
    assert_states_close(got, ref_pool)
    del pool, out
    torch.cuda.empty_cache()
