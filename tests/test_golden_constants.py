"""The workload constants used by the inputs, the library and the oracle
match the values the pages state (tests/golden/kimi_k3_constants.txt)."""
import os

from kda_decode_recurrence_gb300.inputs import BLOCK_CONFIG, DECODE_CONFIGS

HERE = os.path.dirname(os.path.abspath(__file__))


def load():
    vals = {}
    for line in open(os.path.join(HERE, "golden", "kimi_k3_constants.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            name, value = line.split()
            vals[name] = float(value)
    return vals


def test_workloads_use_the_pages_constants():
    g = load()
    for name in ("single", "varlen"):
        assert DECODE_CONFIGS[name].HV == g["num_heads"]
    assert DECODE_CONFIGS["grouped"].HV == g["num_heads"]
    for cfg in DECODE_CONFIGS.values():
        assert cfg.K == cfg.V == g["head_dim"] <= g["max_head_dim"]
    assert DECODE_CONFIGS["varlen"].lower_bound == g["lower_bound"]
    b = BLOCK_CONFIG
    assert b.Kc == g["conv_taps"] and b.lower_bound == g["lower_bound"]
    assert b.rms_norm_eps == g["rms_norm_eps"] and b.l2_eps == g["l2_eps"]
    assert b.K == b.V == g["head_dim"]
    # num_head per rank is a multiple of the head group; 96 / 12 = 8
    assert g["num_heads"] / g["max_tp_for_96_heads"] == 8 and b.nh % 8 == 0
