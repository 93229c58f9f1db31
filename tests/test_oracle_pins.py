"""Pins for the float64 oracle: what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a property
the delta rule must have ("Delta-rule write", Explanation: a key that already
returns the right value writes nothing), a closed form, a special case that
reduces to a library routine (numpy/scipy), or a brute-force restatement of the
naive_recurrent_kda loop on tiny shapes.  The tolerances are float64 rounding
levels: a dropped term, a wrong sign, a transposed operand or a wrong index
moves a result by O(1).
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from oracle import GATE_LOWER_BOUND, GATE_SOFTPLUS

# ---------------------------------------------------------------- helpers


def rand_decode(rng, *, B=3, H=2, HV=4, K=8, V=8, N=6, lengths=(2, 3, 1),
                gate_mode=GATE_SOFTPLUS, lower_bound=-5.0, slots=None):
    lengths = np.asarray(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    d = dict(
        q=rng.standard_normal((T, H, K)), k=rng.standard_normal((T, H, K)),
        v=rng.standard_normal((T, HV, V)), raw_gate=rng.standard_normal((T, HV, K)),
        beta_logits=rng.standard_normal((T, HV)), a_log=np.log(rng.uniform(1, 16, HV)),
        dt_bias=0.1 * rng.standard_normal((HV, K)), cu_seqlens=cu,
        state_pool=0.1 * rng.standard_normal((N, HV, K, V)),
        state_indices=(rng.permutation(N)[:B] if slots is None else np.asarray(slots)).astype(np.int32),
        gate_mode=gate_mode, lower_bound=lower_bound)
    return d


def run(d, **kw):
    args = dict(d)
    args.update(kw)
    return oracle.kda_decode(**args)


def lib_gate(raw, dt, a_log, mode, lb):
    """Gate via library routines: softplus = logaddexp(0, x), sigmoid = expit."""
    x = raw + dt
    if mode == GATE_SOFTPLUS:
        return -np.exp(a_log) * np.logaddexp(0.0, x)
    return lb * expit(np.exp(a_log) * x)


def unit(x):
    return x / np.linalg.norm(x)


# ------------------------------------------------- (a) delta-rule property


@pytest.mark.parametrize("mode", [GATE_SOFTPLUS, GATE_LOWER_BOUND])
def test_a_key_that_already_returns_value_writes_nothing(mode):
    rng = np.random.default_rng(10)
    K = V = 16
    d = rand_decode(rng, B=1, H=1, HV=1, K=K, V=V, N=2, lengths=(1,), gate_mode=mode)
    S = d["state_pool"][d["state_indices"][0], 0]
    g = lib_gate(d["raw_gate"][0, 0], d["dt_bias"][0], d["a_log"][0], mode, d["lower_bound"])
    DS = np.exp(g)[:, None] * S
    kh = unit(d["k"][0, 0])
    d["v"] = (kh @ DS)[None, None, :]            # v := k^T (decayed S)
    for beta_logit in (-1.3, 0.0, 2.7):
        d["beta_logits"] = np.full((1, 1), beta_logit)
        _, pool, st = run(d, l2_eps=0.0)
        assert st == 0
        np.testing.assert_allclose(pool[d["state_indices"][0], 0], DS, rtol=0, atol=1e-14)


# ------------------------------- (b) orthonormal keys, beta = 1, g = 0 recall


def test_b_orthonormal_keys_recall_stored_values():
    rng = np.random.default_rng(11)
    K = V = 8
    m = 5
    keys = np.linalg.qr(rng.standard_normal((K, K)))[0][:, :m].T   # m orthonormal rows
    vals = rng.standard_normal((m, V))
    T = 2 * m
    d = rand_decode(rng, B=1, H=1, HV=1, K=K, V=V, N=1, lengths=(T,),
                    gate_mode=GATE_LOWER_BOUND, lower_bound=0.0)       # g = 0 exactly
    d["state_pool"][:] = 0.0
    d["k"][:m, 0] = keys
    d["v"][:m, 0] = vals
    d["beta_logits"][:m, 0] = 40.0           # sigmoid(40) == 1.0 in float64
    perm = rng.permutation(m)
    d["q"][m:, 0] = keys[perm]
    d["k"][m:, 0] = keys[perm]
    d["beta_logits"][m:, 0] = -800.0         # sigmoid(-800) == 0.0: read without writing
    out, pool, _ = run(d, l2_eps=0.0)
    scale = K ** -0.5
    np.testing.assert_allclose(out[m:, 0], scale * vals[perm], rtol=0, atol=1e-13)
    # the final state holds exactly the m writes: sum_j k_j v_j^T
    np.testing.assert_allclose(pool[0, 0], keys.T @ vals, rtol=0, atol=1e-13)


@pytest.mark.parametrize("mode", [GATE_SOFTPLUS, GATE_LOWER_BOUND])
def test_b_same_token_read_returns_value_for_any_state(mode):
    # With beta = 1 and q = k, q^T S_new = scale * v whatever S and g are:
    # k^T S_new = k^T D S + |k|^2 (v - k^T D S) = v for a unit key.
    rng = np.random.default_rng(12)
    d = rand_decode(rng, B=2, H=2, HV=4, K=16, V=16, N=4, lengths=(3, 2), gate_mode=mode)
    d["q"] = d["k"].copy()
    d["beta_logits"][:] = 40.0
    out, _, _ = run(d, l2_eps=0.0)
    G = 2
    v = d["v"]
    np.testing.assert_allclose(out, 16 ** -0.5 * v, rtol=0, atol=1e-13)
    assert G == d["v"].shape[1] // d["q"].shape[1]


# ------------------------------------------- (c) beta = 0: pure decay


@pytest.mark.parametrize("mode", [GATE_SOFTPLUS, GATE_LOWER_BOUND])
def test_c_beta_zero_is_pure_per_channel_decay(mode):
    rng = np.random.default_rng(13)
    K, V = 8, 12
    d = rand_decode(rng, B=2, H=1, HV=2, K=K, V=V, N=3, lengths=(1, 1), gate_mode=mode)
    d["beta_logits"][:] = -800.0            # sigmoid == 0.0 exactly
    out, pool, _ = run(d, l2_eps=0.0)
    for b in range(2):
        slot = d["state_indices"][b]
        for hv in range(2):
            S0 = d["state_pool"][slot, hv]
            g = lib_gate(d["raw_gate"][b, hv], d["dt_bias"][hv], d["a_log"][hv], mode,
                         d["lower_bound"])
            expect = np.exp(g)[:, None] * S0      # rows (key channels) decay
            np.testing.assert_allclose(pool[slot, hv], expect, rtol=1e-14, atol=0)
            qh = K ** -0.5 * unit(d["q"][b, hv // 2])
            np.testing.assert_allclose(out[b, hv], qh @ expect, rtol=1e-13, atol=1e-15)


def test_c_decay_acts_on_key_rows_not_value_columns():
    # K != V and a gate that differs per key channel: a decay applied along
    # the value axis would not even broadcast to the expected matrix.
    rng = np.random.default_rng(14)
    d = rand_decode(rng, B=1, H=1, HV=1, K=4, V=6, N=1, lengths=(1,))
    d["beta_logits"][:] = -800.0
    d["raw_gate"][0, 0] = np.array([-30.0, 0.0, 1.0, 3.0])
    _, pool, _ = run(d)
    ratio = pool[0, 0] / d["state_pool"][0, 0]
    assert np.allclose(ratio, ratio[:, :1], rtol=1e-13)      # constant along each row
    assert np.ptp(ratio[:, 0]) > 0.1                            # differs between rows


def test_safe_gate_never_amplifies():
    rng = np.random.default_rng(15)
    d = rand_decode(rng, B=1, H=1, HV=1, K=32, V=8, N=1, lengths=(1,),
                    gate_mode=GATE_LOWER_BOUND, lower_bound=-5.0)
    d["raw_gate"] = 10 * rng.standard_normal(d["raw_gate"].shape)
    d["beta_logits"][:] = -800.0
    _, pool, _ = run(d)
    ratio = pool[0, 0][:, 0] / d["state_pool"][0, 0][:, 0]
    assert np.all(ratio <= 1.0) and np.all(ratio >= np.exp(-5.0) * (1 - 1e-15))


# ------------------------- the gate readings, pinned by what the words fix
#
# "KDA Block TKG Kernel API Reference", :param dt_bias: (the bias is added
# before the activation) and :param A_log: (exp(A_log) scales the gate
# pre-activation); "KdaDecode", Default parameters (stable-softplus gate).
# Read together: the pre-activation is exp(A_log) * (raw + dt_bias).  What
# that fixes without restating the formula: at raw = -dt_bias the
# pre-activation is zero for every A_log, so the lower-bound gate is
# lower_bound * sigmoid(0) = lower_bound / 2 and the softplus gate is
# -exp(A_log) * ln 2; for large raw the softplus gate runs along its asymptote
# -exp(A_log) * (raw + dt_bias); at zero pre-activation the lower-bound gate's
# slope in raw is lower_bound * exp(A_log) / 4.  The decay a gate produces is
# read off the oracle's state with beta = 0 (pure decay): row k of the tile is
# multiplied by exp(g_k).


def decay_of(mode, raw, dt, a_log, lb=-5.0):
    """Per-channel exp(g) as the oracle applies it: one token, beta = 0,
    raw gate `raw` [K] and bias `dt` [K] on a single head."""
    K = raw.shape[0]
    rng = np.random.default_rng(5)
    d = rand_decode(rng, B=1, H=1, HV=1, K=K, V=3, N=1, lengths=(1,), gate_mode=mode,
                    lower_bound=lb)
    d["raw_gate"] = raw.reshape(1, 1, K)
    d["dt_bias"] = dt.reshape(1, K)
    d["a_log"] = np.array([a_log])
    d["beta_logits"][:] = -800.0
    d["state_pool"] = 0.5 + rng.uniform(0.0, 1.0, (1, 1, K, 3))
    _, pool, _ = run(d)
    ratio = pool[0, 0] / d["state_pool"][0, 0]
    assert np.allclose(ratio, ratio[:, :1], rtol=1e-15, atol=0)
    return ratio[:, 0]


@pytest.mark.parametrize("a_log", [0.0, np.log(2.5), np.log(16.0)])
@pytest.mark.parametrize("lb", [-5.0, -1.3])
def test_lower_bound_gate_is_half_the_bound_at_zero_preactivation(a_log, lb):
    rng = np.random.default_rng(60)
    dt = 0.3 * rng.standard_normal(8)
    ratio = decay_of(GATE_LOWER_BOUND, -dt, dt, a_log, lb)
    np.testing.assert_allclose(ratio, np.exp(lb / 2), rtol=1e-15)


@pytest.mark.parametrize("a_log,expect", [(0.0, 0.5), (np.log(4.0), 1 / 16), (np.log(16.0), 2.0 ** -16)])
def test_softplus_gate_is_exp_a_log_ln2_at_zero_preactivation(a_log, expect):
    # g = -exp(A_log) ln 2, so exp(g) = 2^-exp(A_log): 1/2, 1/16, 2^-16
    rng = np.random.default_rng(61)
    dt = 0.3 * rng.standard_normal(8)
    ratio = decay_of(GATE_SOFTPLUS, -dt, dt, a_log)
    np.testing.assert_allclose(ratio, expect, rtol=1e-14)


def test_softplus_gate_follows_its_asymptote_for_large_raw():
    # For raw + dt_bias >= 25 the softplus is its argument to 2e-11 relative:
    # g = -exp(A_log) (raw + dt_bias).  Slope and intercept both checked.
    rng = np.random.default_rng(62)
    a = 3.0
    dt = 0.3 * rng.standard_normal(8)
    raw1, raw2 = 25.0 + np.zeros(8) - dt, 31.0 + np.zeros(8) + rng.uniform(0, 1, 8)
    g1 = np.log(decay_of(GATE_SOFTPLUS, raw1, dt, np.log(a)))
    g2 = np.log(decay_of(GATE_SOFTPLUS, raw2, dt, np.log(a)))
    np.testing.assert_allclose((g2 - g1) / (raw2 - raw1), -a, rtol=1e-10)
    np.testing.assert_allclose(g1 + a * raw1, -a * dt, rtol=0, atol=1e-9)


@pytest.mark.parametrize("a_log", [np.log(1.5), np.log(9.0)])
def test_lower_bound_gate_slope_and_limits(a_log):
    rng = np.random.default_rng(63)
    dt = 0.3 * rng.standard_normal(8)
    lb = -5.0
    h = 1e-6
    gp = np.log(decay_of(GATE_LOWER_BOUND, -dt + h, dt, a_log, lb))
    gm = np.log(decay_of(GATE_LOWER_BOUND, -dt - h, dt, a_log, lb))
    np.testing.assert_allclose((gp - gm) / (2 * h), lb * np.exp(a_log) / 4, rtol=1e-6)
    big = np.log(decay_of(GATE_LOWER_BOUND, 60.0 - dt, dt, a_log, lb))
    small = np.log(decay_of(GATE_LOWER_BOUND, -60.0 - dt, dt, a_log, lb))
    np.testing.assert_allclose(big, lb, rtol=1e-15)
    assert np.all(np.abs(small) < 1e-20)


def test_block_forget_gate_bias_joins_the_latent_before_the_scale():
    # One request, W_fb with a single non-zero row, so graw = f_a[0] * W_fb[0];
    # dt_bias set to minus that: the pre-activation is zero and every channel
    # of every head decays by exp(lower_bound / 2), whatever A_log is.
    rng = np.random.default_rng(64)
    p, w = block_small(rng, B=1, nh=3)
    nh, K = 3, 4
    p["W_fb"][1:] = 0.0
    p["A_log"] = np.log(np.array([[1.7, 5.0, 14.0]]))
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True)
    alpha = tr["proj"][0, w["f_a"]]
    p["dt_bias"] = -(alpha * p["W_fb"][0]).reshape(nh, K).T        # dt_bias[d, h]
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True)
    np.testing.assert_array_equal(tr["g"], np.full((1, nh, K), p["lower_bound"] / 2))


# ----------------------------------------- (d) n tokens = n single calls


@pytest.mark.parametrize("mode", [GATE_SOFTPLUS, GATE_LOWER_BOUND])
def test_d_one_call_equals_token_by_token(mode):
    rng = np.random.default_rng(16)
    lengths = (4, 1, 3)
    d = rand_decode(rng, B=3, H=2, HV=4, K=8, V=8, N=5, lengths=lengths, gate_mode=mode)
    out_all, pool_all, _ = run(d)
    cu = d["cu_seqlens"]
    pool = d["state_pool"].copy()
    out_step = np.zeros_like(out_all)
    for b in range(3):
        for t in range(cu[b], cu[b + 1]):
            one = dict(d)
            for name in ("q", "k", "v", "raw_gate", "beta_logits"):
                one[name] = d[name][t:t + 1]
            one["cu_seqlens"] = np.array([0, 1], np.int32)
            one["state_indices"] = d["state_indices"][b:b + 1]
            one["state_pool"] = pool
            o, pool, _ = run(one)
            out_step[t] = o[0]
    assert np.array_equal(out_all, out_step)
    assert np.array_equal(pool_all, pool)


# ------------------------------- (e) brute force: the naive loop restated


def naive_loop(q, k, v, g, beta, scale, S0):
    """The page's naive_recurrent_kda loop restated in float64 torch: all
    heads at once, q and k repeat-interleaved over G, decay then write then
    read.  q, k [B, T, H, K]; v [B, T, HV, V]; g [B, T, HV, K]; beta [B, T, HV]."""
    q, k, v, g, beta, S = (torch.as_tensor(x, dtype=torch.float64) for x in (q, k, v, g, beta, S0))
    G = v.shape[2] // q.shape[2]
    q = q.repeat_interleave(G, dim=2) * scale
    k = k.repeat_interleave(G, dim=2)
    o = torch.zeros_like(v)
    for i in range(q.shape[1]):
        S = S * g[:, i, :, :, None].exp()
        pred = (k[:, i, :, :, None] * S).sum(-2)
        S = S + (beta[:, i, :, None] * k[:, i])[..., None] * (v[:, i] - pred)[:, :, None, :]
        o[:, i] = (q[:, i, :, :, None] * S).sum(-2)
    return o.numpy(), S.numpy()


@pytest.mark.parametrize("KV", [2, 4, 8])
@pytest.mark.parametrize("H,G", [(1, 1), (1, 2), (2, 1), (2, 2)])
@pytest.mark.parametrize("mode", [GATE_SOFTPLUS, GATE_LOWER_BOUND])
def test_e_brute_force_tiny(KV, H, G, mode):
    rng = np.random.default_rng(100 + KV * 10 + H * 3 + G + mode * 50)
    Bn, n = 2, 5
    HV = H * G
    d = rand_decode(rng, B=Bn, H=H, HV=HV, K=KV, V=KV, N=Bn + 2, lengths=(n,) * Bn,
                    gate_mode=mode)
    eps = 1e-6
    out, pool, _ = run(d, l2_eps=eps)
    # activated inputs for the naive loop
    T = Bn * n
    qn = d["q"] / np.sqrt((d["q"] ** 2).sum(-1, keepdims=True) + eps)
    kn = d["k"] / np.sqrt((d["k"] ** 2).sum(-1, keepdims=True) + eps)
    x = torch.as_tensor(d["raw_gate"] + d["dt_bias"][None])
    A = torch.as_tensor(np.exp(d["a_log"]))[None, :, None]
    if mode == GATE_SOFTPLUS:
        g = (-A * torch.nn.functional.softplus(x)).numpy()
    else:
        g = (d["lower_bound"] * torch.sigmoid(A * x)).numpy()
    beta = torch.sigmoid(torch.as_tensor(d["beta_logits"])).numpy()
    rs = lambda a: a.reshape((Bn, n) + a.shape[1:])  # noqa: E731
    S0 = d["state_pool"][d["state_indices"]]
    o_ref, S_ref = naive_loop(rs(qn), rs(kn), rs(d["v"]), rs(g), rs(beta), KV ** -0.5, S0)
    np.testing.assert_allclose(out.reshape(Bn, n, HV, KV), o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(pool[d["state_indices"]], S_ref, rtol=0, atol=1e-12)
    assert T == out.shape[0]


# ------------------------------------------------------- extra pins


def test_read_after_write_from_zero_state():
    # S0 = 0, one token: S1 = beta k v^T, o = beta (q.k) v with the scale.
    rng = np.random.default_rng(17)
    K, V = 8, 8
    d = rand_decode(rng, B=1, H=1, HV=1, K=K, V=V, N=1, lengths=(1,))
    d["state_pool"][:] = 0.0
    out, pool, _ = run(d, l2_eps=0.0)
    beta = expit(d["beta_logits"][0, 0])
    qh, kh = K ** -0.5 * unit(d["q"][0, 0]), unit(d["k"][0, 0])
    np.testing.assert_allclose(out[0, 0], beta * (qh @ kh) * d["v"][0, 0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(pool[0, 0], beta * np.outer(kh, d["v"][0, 0]), rtol=1e-13, atol=1e-16)


def test_gva_equals_explicit_repeat_interleave():
    rng = np.random.default_rng(18)
    d = rand_decode(rng, B=3, H=3, HV=6, K=8, V=8, N=4, lengths=(2, 1, 2))
    out_g, pool_g, _ = run(d)
    e = dict(d)
    e["q"] = np.repeat(d["q"], 2, axis=1)     # value head hv reads key head hv // 2
    e["k"] = np.repeat(d["k"], 2, axis=1)
    out_e, pool_e, _ = run(e)
    assert np.array_equal(out_g, out_e) and np.array_equal(pool_g, pool_e)
    f = dict(d)
    f["q"] = np.tile(d["q"], (1, 2, 1))       # the wrong mapping hv % H must differ
    f["k"] = np.tile(d["k"], (1, 2, 1))
    out_f, _, _ = run(f)
    assert np.abs(out_f - out_g).max() > 1e-3


def test_query_and_key_are_scale_invariant():
    rng = np.random.default_rng(19)
    d = rand_decode(rng)
    out, pool, _ = run(d, l2_eps=0.0)
    for name in ("q", "k"):
        e = dict(d)
        e[name] = d[name] * 7.5
        out2, pool2, _ = run(e, l2_eps=0.0)
        np.testing.assert_allclose(out2, out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(pool2, pool, rtol=0, atol=1e-12)


def test_zero_query_and_key_give_finite_results():
    rng = np.random.default_rng(20)
    d = rand_decode(rng, B=1, H=1, HV=1, N=1, lengths=(2,))
    d["q"][0] = 0.0
    d["k"][1] = 0.0
    out, pool, _ = run(d)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(pool))
    assert np.all(out[0] == 0.0)


def test_slot_routing_permutation_and_untouched_slots():
    rng = np.random.default_rng(21)
    N = 9
    d = rand_decode(rng, B=4, H=2, HV=2, K=8, V=8, N=N, lengths=(1, 2, 1, 3))
    # distinct values in every slot so a misrouted slot is an O(1) error
    d["state_pool"] += np.arange(N)[:, None, None, None]
    out, pool, st = run(d)
    assert st == 0
    used = set(d["state_indices"].tolist())
    for s in range(N):
        if s not in used:
            assert np.array_equal(pool[s], d["state_pool"][s])
    # permute requests (with their tokens and slots)
    perm = np.array([2, 0, 3, 1])
    cu = d["cu_seqlens"]
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in perm])
    e = dict(d)
    for name in ("q", "k", "v", "raw_gate", "beta_logits"):
        e[name] = d[name][rows]
    lengths = np.diff(cu)[perm]
    e["cu_seqlens"] = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    e["state_indices"] = d["state_indices"][perm]
    out_p, pool_p, _ = run(e)
    assert np.array_equal(out_p, out[rows]) and np.array_equal(pool_p, pool)


def test_padded_and_invalid_slots_and_seqlens():
    rng = np.random.default_rng(22)
    d = rand_decode(rng, B=3, H=1, HV=2, K=4, V=4, N=4, lengths=(1, 2, 1), slots=(1, -1, 7))
    init = np.full((4, 2, 4), 9.0)
    out, pool, st = run(d, output=init)
    assert st == oracle.BAD_SLOT
    assert np.all(out[1:4] == 0.0)                       # padded (-1) and bad (7) rows zeroed
    assert np.array_equal(pool[[0, 2, 3]], d["state_pool"][[0, 2, 3]])
    assert not np.array_equal(pool[1], d["state_pool"][1])
    e = dict(d)
    e["state_indices"] = np.array([1, 2, 3], np.int32)
    e["cu_seqlens"] = np.array([0, 3, 2, 4], np.int32)   # decreasing range for request 1
    out2, pool2, st2 = run(e, output=init)
    assert st2 == oracle.BAD_SEQLEN
    assert np.array_equal(pool2[2], d["state_pool"][2])  # skipped request untouched
    e["cu_seqlens"] = np.array([0, 1, 3, 5], np.int32)   # last entry past T
    _, _, st3 = run(e, output=init)
    assert st3 == oracle.BAD_SEQLEN


def test_empty_request_leaves_state_bit_identical():
    rng = np.random.default_rng(23)
    d = rand_decode(rng, B=3, H=1, HV=2, K=4, V=4, N=4, lengths=(2, 0, 1))
    _, pool, st = run(d)
    assert st == 0
    s = d["state_indices"][1]
    assert np.array_equal(pool[s], d["state_pool"][s])


# ----------------------------------------------------------- block pins


def block_small(rng, B=2, n=1, Hd=16, nh=2, K=4, Kc=4, gamma=False):
    V = K
    w = oracle.oracle.block_widths(nh, K, V)
    I = w["I"]
    return dict(
        hidden=rng.standard_normal((B, n, Hd)),
        gamma_in=(rng.uniform(0.5, 1.5, (1, Hd)) if gamma else np.ones((1, Hd))),
        W_in=0.3 * rng.standard_normal((Hd, I)), W_fb=0.3 * rng.standard_normal((K, K * nh)),
        W_gb=0.3 * rng.standard_normal((K, V * nh)),
        conv_w=0.5 * rng.standard_normal((3, Kc, K * nh)),
        A_log=np.log(rng.uniform(1, 16, (1, nh))), dt_bias=0.1 * rng.standard_normal((K, nh)),
        gamma_o=rng.uniform(0.5, 1.5, (1, V)), W_o=0.3 * rng.standard_normal((V * nh, Hd)),
        S=0.1 * rng.standard_normal((B, nh, K, V)),
        conv_state=0.5 * rng.standard_normal((B, 3, K * nh, Kc - 1)),
        scale=K ** -0.5, lower_bound=-5.0, rms_norm_eps=1e-5, l2_eps=1e-6), w


def silu(x):
    return x * expit(x)


def test_block_input_rmsnorm_and_projection():
    rng = np.random.default_rng(30)
    p, w = block_small(rng, gamma=True)
    p["rms_norm_eps"] = 0.0
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True)
    xh = tr["xhat"] / p["gamma_in"]
    np.testing.assert_allclose((xh ** 2).mean(-1), 1.0, rtol=1e-14)     # unit RMS
    x = p["hidden"].reshape(-1, p["hidden"].shape[-1])
    np.testing.assert_allclose(xh * np.linalg.norm(x, axis=1, keepdims=True) / np.sqrt(x.shape[1]),
                               x, rtol=1e-13)
    np.testing.assert_allclose(tr["proj"], tr["xhat"] @ p["W_in"], rtol=1e-12, atol=1e-13)


def test_block_conv_layout_and_state_shift():
    rng = np.random.default_rng(31)
    p, w = block_small(rng)
    nh, K = 2, 4
    Kc = p["conv_w"].shape[1]
    # newest tap only: y = SiLU(projection), exposing each stream's channel order
    p["conv_w"][:] = 0.0
    p["conv_w"][:, Kc - 1, :] = 1.0
    _, _, cs, tr = oracle.kda_block_tkg(**p, trace=True)
    P = tr["proj"]
    for h in range(nh):
        for dd in range(K):
            np.testing.assert_allclose(tr["qc"][:, h, dd], silu(P[:, w["q"] + dd * nh + h]), rtol=1e-14)
            np.testing.assert_allclose(tr["kc"][:, h, dd], silu(P[:, w["k"] + dd * nh + h]), rtol=1e-14)
            np.testing.assert_allclose(tr["vc"][:, h, dd], silu(P[:, w["v"] + h * K + dd]), rtol=1e-14)
    # window shift: [old1, old2, new] for every stream
    old = p["conv_state"]
    np.testing.assert_array_equal(cs[..., :Kc - 2], old[..., 1:])
    CQ = nh * K
    np.testing.assert_array_equal(cs[:, 0, :, -1], P[:, w["q"]:w["q"] + CQ])
    np.testing.assert_array_equal(cs[:, 1, :, -1], P[:, w["k"]:w["k"] + CQ])
    np.testing.assert_array_equal(cs[:, 2, :, -1], P[:, w["v"]:w["v"] + CQ])
    # oldest tap only: y = SiLU(conv_state[..., 0])
    p["conv_w"][:] = 0.0
    p["conv_w"][:, 0, :] = 1.0
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True)
    for h in range(nh):
        np.testing.assert_allclose(tr["qc"][:, h, 1], silu(old[:, 0, 1 * nh + h, 0]), rtol=1e-14)
        np.testing.assert_allclose(tr["vc"][:, h, 1], silu(old[:, 2, h * K + 1, 0]), rtol=1e-14)


def test_block_conv_general_taps_match_numpy_convolution():
    rng = np.random.default_rng(32)
    p, w = block_small(rng)
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True)
    P = tr["proj"]
    nh, K = 2, 4
    for b in range(2):
        for dd in range(K):
            for h in range(nh):
                c = dd * nh + h
                window = np.concatenate([p["conv_state"][b, 0, c], [P[b, w["q"] + c]]])
                # correlation with taps ordered oldest..newest == np.convolve with reversed taps
                y = np.convolve(window, p["conv_w"][0, ::-1, c], mode="valid")[0]
                np.testing.assert_allclose(tr["qc"][b, h, dd], silu(y), rtol=1e-13)


def test_block_gate_latents_layouts():
    rng = np.random.default_rng(33)
    p, w = block_small(rng)
    nh, K = 2, 4
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True)
    P = tr["proj"]
    fa = P[:, w["f_a"]:w["f_a"] + K]
    ga = P[:, w["g_a"]:w["g_a"] + K]
    gb = fa @ p["W_fb"]
    zb = ga @ p["W_gb"]
    for h in range(nh):
        for dd in range(K):
            np.testing.assert_allclose(tr["graw"][:, h, dd], gb[:, h * K + dd], rtol=1e-13)
            np.testing.assert_allclose(tr["z"][:, h, dd], zb[:, dd * nh + h], rtol=1e-13)
            expect_g = p["lower_bound"] * expit(np.exp(p["A_log"][0, h]) *
                                                (gb[:, h * K + dd] + p["dt_bias"][dd, h]))
            np.testing.assert_allclose(tr["g"][:, h, dd], expect_g, rtol=1e-13)
    np.testing.assert_allclose(tr["beta"], expit(P[:, w["beta"]:w["beta"] + nh]), rtol=1e-14)


def test_block_recurrence_matches_decode_oracle():
    rng = np.random.default_rng(34)
    p, w = block_small(rng, B=3, nh=3)
    out, S_new, _, tr = oracle.kda_block_tkg(**p, trace=True)
    B, nh, K = 3, 3, 4
    P = tr["proj"]
    o, pool, st = oracle.kda_decode(
        q=tr["qc"], k=tr["kc"], v=tr["vc"], raw_gate=tr["graw"],
        beta_logits=P[:, w["beta"]:w["beta"] + nh], a_log=p["A_log"][0],
        dt_bias=p["dt_bias"].T, cu_seqlens=np.arange(B + 1), state_pool=p["S"],
        state_indices=np.arange(B), gate_mode=GATE_LOWER_BOUND, lower_bound=p["lower_bound"],
        scale=p["scale"], l2_eps=p["l2_eps"])
    assert st == 0
    np.testing.assert_allclose(tr["o"], o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(S_new, pool, rtol=0, atol=1e-14)


def test_block_gated_norm_and_identity_output_projection():
    rng = np.random.default_rng(35)
    nh, K = 2, 4
    p, w = block_small(rng, Hd=nh * K, nh=nh, K=K)
    p["W_o"] = np.eye(nh * K)
    out, _, _, tr = oracle.kda_block_tkg(**p, trace=True)
    np.testing.assert_array_equal(out.reshape(-1, nh * K), tr["on"].reshape(-1, nh * K))
    o = tr["o"]
    rms = np.sqrt((o ** 2).mean(-1, keepdims=True) + p["rms_norm_eps"])
    np.testing.assert_allclose(tr["on"], o / rms * p["gamma_o"][0] * expit(tr["z"]), rtol=1e-13)


def test_block_gated_norm_unit_rms_when_gate_open():
    rng = np.random.default_rng(36)
    p, w = block_small(rng)
    p["gamma_o"][:] = 1.0
    p["rms_norm_eps"] = 0.0
    K = 4
    # make g_a huge so sigmoid(z) == 1 to double precision where z > 40
    p["W_in"][:, w["g_a"]:w["g_a"] + K] = 0.0
    p["W_in"][0, w["g_a"]] = 1e4
    p["W_gb"][:] = 0.0
    p["W_gb"][0, :] = 1.0
    p["hidden"][..., 0] = np.abs(p["hidden"][..., 0]) + 1.0
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True)
    assert np.all(tr["z"] > 40)
    np.testing.assert_allclose((tr["on"] ** 2).mean(-1), 1.0, rtol=1e-13)


def test_block_multi_token_equals_sequential_single_tokens():
    rng = np.random.default_rng(37)
    p, w = block_small(rng, B=2, n=3)
    out, S_new, cs_new = oracle.kda_block_tkg(**p)
    S, cs = p["S"], p["conv_state"]
    for j in range(3):
        q = dict(p)
        q["hidden"] = p["hidden"][:, j:j + 1]
        q["S"], q["conv_state"] = S, cs
        o1, S, cs = oracle.kda_block_tkg(**q)
        assert np.array_equal(o1[:, 0], out[:, j])
    assert np.array_equal(S, S_new) and np.array_equal(cs, cs_new)


# ------------------------------------------ the output gate, per setting
#
# "KDA Block TKG Kernel API Reference", Background: a "gated" output RMSNorm,
# with no activation named.  Sigmoid is the default reading and swish
# (z * sigmoid(z)) the alternative; each setting is pinned by its values at
# z = 0 (W_gb = 0) and at z >> 0, where the norm alone is o / rms * gamma_o.


def open_gate_block(rng, z_big):
    p, w = block_small(rng)
    p["rms_norm_eps"] = 0.0
    K = 4
    if z_big:
        p["W_in"][:, w["g_a"]:w["g_a"] + K] = 0.0
        p["W_in"][0, w["g_a"]] = 1e4
        p["W_gb"][:] = 0.0
        p["W_gb"][0, :] = 1.0
        p["hidden"][..., 0] = np.abs(p["hidden"][..., 0]) + 1.0
    else:
        p["W_gb"][:] = 0.0
    return p


@pytest.mark.parametrize("gate,at_zero", [("sigmoid", 0.5), ("swish", 0.0)])
def test_output_gate_at_zero(gate, at_zero):
    p = open_gate_block(np.random.default_rng(70), z_big=False)
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True, out_gate=gate)
    assert np.all(tr["z"] == 0.0)
    norm = tr["o"] / np.sqrt((tr["o"] ** 2).mean(-1, keepdims=True)) * p["gamma_o"][0]
    np.testing.assert_allclose(tr["on"], at_zero * norm, rtol=1e-13, atol=0)


@pytest.mark.parametrize("gate", ["sigmoid", "swish"])
def test_output_gate_wide_open(gate):
    p = open_gate_block(np.random.default_rng(71), z_big=True)
    _, _, _, tr = oracle.kda_block_tkg(**p, trace=True, out_gate=gate)
    assert np.all(tr["z"] > 40)
    norm = tr["o"] / np.sqrt((tr["o"] ** 2).mean(-1, keepdims=True)) * p["gamma_o"][0]
    # sigmoid(z) == 1 and z * sigmoid(z) == z to double precision here
    expect = norm if gate == "sigmoid" else tr["z"] * norm
    np.testing.assert_allclose(tr["on"], expect, rtol=1e-13, atol=0)
