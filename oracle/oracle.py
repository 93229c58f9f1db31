"""ctypes wrapper around the float64 C oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Inputs are numpy arrays
of any float dtype; they are widened to float64 here (bf16/fp32 values widen
exactly) and the oracle computes in float64 throughout.

The C source is compiled with the host C compiler into ``oracle/_build`` on
first use (or by ``build()``), so the same checker runs on any host CPU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# Status bits and gate modes, as the oracle's own C source defines them.
BAD_SLOT = 1
BAD_SEQLEN = 2
GATE_SOFTPLUS = 0
GATE_LOWER_BOUND = 1
OUT_GATES = {"sigmoid": 0, "swish": 1}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``_build/liboracle.so`` (plain C, -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps every product and sum as written (no fused
    # multiply-add contraction), so results are the same on x86 and Arm.
    cmd = ["cc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Trace(ctypes.Structure):
    _fields_ = [(name, ctypes.POINTER(ctypes.c_double)) for name in
                ("xhat", "proj", "qc", "kc", "vc", "graw", "g", "beta", "o", "z", "on")]


def configure(lib):
    """Declare the C signatures on a loaded copy of the oracle library."""
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    c_int, c_double = ctypes.c_int, ctypes.c_double
    lib.oracle_kda_decode.restype = c_int
    lib.oracle_kda_decode.argtypes = (
        [dp, dp, dp, dp, dp, dp, dp, dp, ip, dp, ip, c_int, c_double, c_double,
         c_double] + [c_int] * 7 + [ip])
    lib.oracle_kda_block_tkg.restype = c_int
    lib.oracle_kda_block_tkg.argtypes = (
        [dp] * 11 + [dp, dp] + [c_double] * 4 + [c_int] * 8 + [ctypes.POINTER(_Trace)])
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # KDA_ORACLE_LIB points the wrapper at another build of the same
            # source; the mutation tests use it to load deliberately broken
            # copies and check that the pins reject them.
            path = os.environ.get("KDA_ORACLE_LIB") or build()
            _lib = configure(ctypes.CDLL(path))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def kda_decode(q, k, v, raw_gate, beta_logits, a_log, dt_bias, cu_seqlens, state_pool,
               state_indices, gate_mode=GATE_SOFTPLUS, lower_bound=-5.0, scale=None,
               l2_eps=1e-6, output=None):
    """Float64 decode recurrence.  Shapes (leading batch-of-1 axis optional):
    q, k [T, H, K]; v [T, HV, V]; raw_gate [T, HV, K]; beta_logits [T, HV];
    a_log [HV]; dt_bias [HV, K]; cu_seqlens [B+1]; state_pool [N, HV, K, V];
    state_indices [B].

    Returns ``(output [T, HV, V], new_state_pool, status)``; the input pool is
    not modified (the oracle advances a float64 copy).  ``output`` may pass an
    initial output array (rows no request covers keep its values; default
    zeros).
    """
    q = _f64(q); k = _f64(k); v = _f64(v)
    if q.ndim == 4:
        q, k, v = q[0], k[0], v[0]
        raw_gate = np.asarray(raw_gate)[0]
        beta_logits = np.asarray(beta_logits)[0]
    T, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    raw_gate = _f64(raw_gate).reshape(T, HV, K)
    beta_logits = _f64(beta_logits).reshape(T, HV)
    a_log = _f64(a_log).reshape(HV)
    dt_bias = _f64(dt_bias).reshape(HV, K)
    cu = _i32(cu_seqlens)
    idx = _i32(state_indices)
    B = idx.shape[0]
    assert cu.shape[0] == B + 1
    pool = _f64(state_pool).copy()
    N = pool.shape[0]
    assert pool.shape == (N, HV, K, V)
    out = np.zeros((T, HV, V)) if output is None else _f64(output).copy()
    if scale is None:
        scale = K ** -0.5
    status = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_kda_decode(
        _dp(out), _dp(q), _dp(k), _dp(v), _dp(raw_gate), _dp(beta_logits), _dp(a_log),
        _dp(dt_bias), _ip(cu), _dp(pool), _ip(idx), int(gate_mode), float(lower_bound),
        float(scale), float(l2_eps), B, T, H, HV, K, V, N, _ip(status))
    if rc != 0:
        raise ValueError(f"oracle_kda_decode rejected its arguments (rc={rc})")
    return out, pool, int(status[0])


def block_widths(nh: int, K: int, V: int) -> dict:
    """Column offsets of the fused projection q | k | v | g_a | beta | f_a."""
    CQ, CV = K * nh, V * nh
    off = {"q": 0, "k": CQ, "v": 2 * CQ, "g_a": 2 * CQ + CV}
    off["beta"] = off["g_a"] + K
    off["f_a"] = off["beta"] + nh
    off["I"] = off["f_a"] + K
    return off


def kda_block_tkg(hidden, gamma_in, W_in, W_fb, W_gb, conv_w, A_log, dt_bias, gamma_o, W_o,
                  S, conv_state, scale, lower_bound, rms_norm_eps=1e-5, l2_eps=1e-6,
                  trace=False, out_gate="sigmoid"):
    """Float64 fused KDA block.  Shapes: hidden [B, n, Hd]; gamma_in [1, Hd];
    W_in [Hd, I]; W_fb [K, K*nh]; W_gb [K, V*nh]; conv_w [3, Kc, K*nh];
    A_log [1, nh]; dt_bias [K, nh]; gamma_o [1, V]; W_o [V*nh, Hd];
    S [B, nh, K, V]; conv_state [B, 3, K*nh, Kc-1].

    ``out_gate`` is the output-gate activation, "sigmoid" (default) or
    "swish".  Returns ``(out [B, n, Hd], S_new, conv_state_new)`` and, with
    ``trace=True``, a dict of the block's intermediates as a fourth item.
    The inputs are not modified.
    """
    hidden = _f64(hidden)
    B, n, Hd = hidden.shape
    S = _f64(S).copy()
    _, nh, K, V = S.shape
    conv_state = _f64(conv_state).copy()
    Kc = conv_state.shape[-1] + 1
    I = block_widths(nh, K, V)["I"]
    W_in = _f64(W_in)
    assert W_in.shape == (Hd, I), (W_in.shape, (Hd, I))
    args = [_f64(gamma_in).reshape(Hd), W_in, _f64(W_fb).reshape(K, K * nh),
            _f64(W_gb).reshape(K, V * nh), _f64(conv_w).reshape(3, Kc, K * nh),
            _f64(A_log).reshape(nh), _f64(dt_bias).reshape(K, nh), _f64(gamma_o).reshape(V),
            _f64(W_o).reshape(V * nh, Hd)]
    out = np.zeros((B, n, Hd))
    tr_arrays = None
    tr_ptr = None
    if trace:
        R = B * n
        tr_arrays = {"xhat": np.zeros((R, Hd)), "proj": np.zeros((R, I)),
                     "qc": np.zeros((R, nh, K)), "kc": np.zeros((R, nh, K)),
                     "vc": np.zeros((R, nh, V)), "graw": np.zeros((R, nh, K)),
                     "g": np.zeros((R, nh, K)), "beta": np.zeros((R, nh)),
                     "o": np.zeros((R, nh, V)), "z": np.zeros((R, nh, V)),
                     "on": np.zeros((R, nh, V))}
        tr = _Trace(**{name: _dp(arr) for name, arr in tr_arrays.items()})
        tr_ptr = ctypes.pointer(tr)
    rc = _load().oracle_kda_block_tkg(
        _dp(out), _dp(hidden), *[_dp(a) for a in args], _dp(S), _dp(conv_state),
        float(scale), float(lower_bound), float(rms_norm_eps), float(l2_eps),
        B, n, Hd, nh, K, V, Kc, OUT_GATES[out_gate], tr_ptr)
    if rc != 0:
        raise ValueError(f"oracle_kda_block_tkg rejected its arguments (rc={rc})")
    if trace:
        return out, S, conv_state, tr_arrays
    return out, S, conv_state
