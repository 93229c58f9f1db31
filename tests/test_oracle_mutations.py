"""The oracle's pins must reject plausible mistakes.

Each case plants one mistake in a copy of ``oracle/kda_oracle.c`` (on the CPU,
in a temporary directory), builds it, and runs the pin suite against it in a
subprocess; the suite must fail.  This is how the pins are shown to pin
something: a dropped term, a flipped sign, a transposed operand, a wrong index
or a wrong order each has to trip at least one of them.
"""
import concurrent.futures as cf
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
    ("output_gate_dropped", "on[(size_t)h * V + d] = o[d] * oinv * gamma_o[d] * output_gate(zz, out_gate);",
     "on[(size_t)h * V + d] = o[d] * oinv * gamma_o[d];"),
    ("output_norm_dropped", "on[(size_t)h * V + d] = o[d] * oinv * gamma_o[d] * output_gate(zz, out_gate);",
     "on[(size_t)h * V + d] = o[d] * gamma_o[d] * output_gate(zz, out_gate);"),
    # the other readings of the gate words: dt_bias added after the exp(A_log)
    # scale, or the scale taken inside the softplus
    ("gate_bias_after_scale_lower_bound", "return lower_bound * sigmoid(exp(a_log) * x);",
     "return lower_bound * sigmoid(exp(a_log) * raw + dt_bias);"),
    ("gate_bias_after_scale_softplus", "return -exp(a_log) * softplus(x);",
     "return -softplus(exp(a_log) * raw + dt_bias);"),
    ("gate_scale_inside_softplus", "return -exp(a_log) * softplus(x);",
     "return -softplus(exp(a_log) * x);"),
    ("block_gate_bias_after_scale", "sigmoid(exp(A_log[h]) * (acc + dt_bias[(size_t)d * nh + h]))",
     "sigmoid(exp(A_log[h]) * acc + dt_bias[(size_t)d * nh + h])"),
    # the two output-gate settings swapped for one another
    ("output_gate_swish_as_default", "  return sigmoid(z);\n}", "  return z * sigmoid(z);\n}"),
    ("output_gate_swish_setting_is_sigmoid", "if (out_gate == ORACLE_OUT_GATE_SWISH) return z * sigmoid(z);",
     "if (out_gate == ORACLE_OUT_GATE_SWISH) return sigmoid(z);"),
]


def _build_mutant(tmp_dir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/absent"
    path = os.path.join(tmp_dir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmp_dir, f"{name}.so")
    subprocess.run(["cc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                    path, "-o", lib, "-lm"], check=True)
    return lib


def _run_pins(lib):
    env = dict(os.environ, KDA_ORACLE_LIB=str(lib))
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    """Every mutant built and run against the pin suite, several at a time
    (each run is its own subprocess)."""
    tmp = str(tmp_path_factory.mktemp("mutants"))

    def one(m):
        name, old, new = m
        return name, _run_pins(_build_mutant(tmp, name, old, new))

    workers = max(1, min(len(MUTANTS), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        return dict(ex.map(one, MUTANTS))


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_reject_mutant(mutant_results, name):
    r = mutant_results[name]
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
