"""The oracle's pins must reject plausible mistakes.

Each case plants one mistake in a copy of ``oracle/kda_oracle.c`` (on the CPU,
in a temporary directory), builds it, and runs the pin suite against it in a
subprocess; the suite must fail.  This is how the pins are shown to pin
something: a dropped term, a flipped sign, a transposed operand, a wrong index
or a wrong order each has to trip at least one of them.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")

# (name, text in the oracle, replacement)
MUTANTS = [
    ("sign_of_correction", "u[j] = v[j] - ks;", "u[j] = v[j] + ks;"),
    ("transposed_key_read", "ks += kh[i] * S[i * V + j];", "ks += kh[i] * S[j * V + i];"),
    ("dropped_decay", "S[i * V + j] *= d;", "S[i * V + j] *= 1.0;"),
    ("decay_on_value_axis", "double d = exp(g[i]);\n    for (int j = 0; j < V; ++j) S[i * V + j] *= d;",
     "for (int j = 0; j < V; ++j) S[i * V + j] *= exp(g[j % K]);"),
    ("dropped_beta", "S[i * V + j] += beta * kh[i] * u[j];", "S[i * V + j] += kh[i] * u[j];"),
    ("read_with_key", "acc += qh[i] * S[i * V + j];", "acc += kh[i] * S[i * V + j];"),
    ("gate_sign", "return -exp(a_log) * softplus(x);", "return exp(a_log) * softplus(x);"),
    ("gate_without_a_log", "return lower_bound * sigmoid(exp(a_log) * x);",
     "return lower_bound * sigmoid(x);"),
    ("no_query_scale", "l2_normalise(qh, q + ((size_t)t * H + h) * K, K, l2_eps, scale);",
     "l2_normalise(qh, q + ((size_t)t * H + h) * K, K, l2_eps, 1.0);"),
    ("no_key_norm", "for (int i = 0; i < n; ++i) out[i] = x[i] * inv * mul;",
     "for (int i = 0; i < n; ++i) out[i] = x[i] * (mul == 1.0 ? 1.0 : inv * mul);"),
    ("gva_modulo", "int h = hv / G;", "int h = hv % H;"),
    ("padded_rows_not_zeroed", "for (int j = 0; j < V; ++j) output[((size_t)t * HV + hv) * V + j] = 0.0;",
     "for (int j = 0; j < V; ++j) (void)0;"),
    ("rmsnorm_no_mean", "  ms /= Hd;\n", "\n"),
    ("q_conv_head_outer", "tmpq[d] = y[0 * (size_t)CS + (size_t)d * nh + h];",
     "tmpq[d] = y[0 * (size_t)CS + (size_t)h * K + d];"),
    ("v_conv_channel_outer", "vv[d] = y[2 * (size_t)CS + (size_t)h * V + d];",
     "vv[d] = y[2 * (size_t)CS + (size_t)d * nh + h];"),
    ("conv_tap_reversed", "acc += conv_w[((size_t)s * Kc + t) * CS + c] * cs[t];",
     "acc += conv_w[((size_t)s * Kc + (Kc - 1 - t)) * CS + c] * cs[t];"),
    ("conv_state_not_shifted", "for (int t = 0; t + 1 < Kc - 1; ++t) cs[t] = cs[t + 1];", ""),
    ("no_silu", "y[(size_t)s * CS + c] = acc * sigmoid(acc);", "y[(size_t)s * CS + c] = acc;"),
    ("fb_channel_outer", "double acc = graw[(size_t)h * K + d];", "double acc = graw[(size_t)d * nh + h];"),
    ("dt_bias_transposed", "(acc + dt_bias[(size_t)d * nh + h])", "(acc + dt_bias[(size_t)h * K + d])"),
    ("gb_head_outer", "double zz = zall[(size_t)d * nh + h];", "double zz = zall[(size_t)h * V + d];"),
    ("output_gate_dropped", "on[(size_t)h * V + d] = o[d] * oinv * gamma_o[d] * sigmoid(zz);",
     "on[(size_t)h * V + d] = o[d] * oinv * gamma_o[d];"),
    ("output_norm_dropped", "on[(size_t)h * V + d] = o[d] * oinv * gamma_o[d] * sigmoid(zz);",
     "on[(size_t)h * V + d] = o[d] * gamma_o[d] * sigmoid(zz);"),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/absent"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"{name}.so"
    subprocess.run(["cc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                    str(path), "-o", str(lib), "-lm"], check=True)
    return lib


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    lib = _build_mutant(tmp_path, name, old, new)
    env = dict(os.environ, KDA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
