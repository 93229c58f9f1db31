"""The C ABI (include/kda.h): the library loads, exports every declared symbol,
and rejects bad arguments on the host before any launch.  No GPU needed: every
call here returns from host validation."""
import ctypes
import os
import re

import pytest

from kda_decode_recurrence_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

KDA_OK, ERR_NULL, ERR_SHAPE, ERR_UNSUP, ERR_ENUM, ERR_CUDA, ERR_ALIGN, ERR_VALUE, ERR_WS = \
    0, -1, -2, -3, -4, -5, -6, -7, -8


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_header_declares_the_documented_calls():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.kda_version().decode().startswith("kda-gb300")


@pytest.mark.parametrize("variant", sorted(build.VARIANTS))
def test_variant_library_exports_every_declared_symbol(lib, variant):
    vlib = _lib.load_variant(variant)
    for name in declared_functions():
        assert hasattr(vlib, name), name
    assert vlib.kda_version().decode() == lib.kda_version().decode()


def test_testhooks_variant_exports_its_hooks():
    vlib = _lib.load_variant("testhooks")
    for name in ("kda_test_set_decode_hooks", "kda_test_set_prefill_hooks"):
        assert hasattr(vlib, name), name


def test_status_strings(lib):
    for code in _lib.STATUS:
        s = lib.kda_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.kda_status_string(12345).decode() == "unknown status"


# A fake but 256-byte-aligned "device" address: validation never dereferences.
P = 0x10000


def decode_args(**kw):
    a = dict(output=P, q=P, k=P, v=P, raw_gate=P, beta_logits=P, a_log=P, dt_bias=P,
             cu_seqlens=P, state_pool=P, state_indices=P, gate_mode=0, lower_bound=-5.0,
             B=2, T=3, H=2, HV=4, K=128, V=128, max_slots=8, dev_status=None, stream=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,expect", [
    ({"B": -1}, ERR_SHAPE), ({"T": -1}, ERR_SHAPE), ({"H": 0}, ERR_SHAPE),
    ({"HV": 3}, ERR_SHAPE), ({"max_slots": 0}, ERR_SHAPE),
    ({"K": 64}, ERR_UNSUP), ({"V": 96}, ERR_UNSUP),
    ({"gate_mode": 2}, ERR_ENUM), ({"gate_mode": -1}, ERR_ENUM),
    ({"gate_mode": 1, "lower_bound": float("nan")}, ERR_VALUE),
    ({"gate_mode": 1, "lower_bound": 0.5}, ERR_VALUE),
    ({"state_pool": None}, ERR_NULL), ({"q": None}, ERR_NULL), ({"cu_seqlens": None}, ERR_NULL),
    ({"output": None}, ERR_NULL), ({"state_indices": None}, ERR_NULL),
    ({"state_pool": P + 8}, ERR_ALIGN), ({"output": P + 4}, ERR_ALIGN),
    ({"raw_gate": P + 8}, ERR_ALIGN), ({"q": P + 2}, ERR_ALIGN),
    ({"B": 0}, KDA_OK),                          # nothing to do: no launch
])
def test_decode_host_validation(lib, kw, expect):
    assert lib.kda_decode(*decode_args(**kw)) == expect


def test_decode_token_pointers_may_be_null_without_tokens(lib):
    # T == 0 with B == 0 returns before any launch
    args = decode_args(B=0, T=0, q=None, k=None, v=None, raw_gate=None, beta_logits=None,
                       output=None)
    assert lib.kda_decode(*args) == KDA_OK


def block_args(**kw):
    a = dict(out=P, hidden=P, gamma_in=P, W_in=P, W_fb=P, W_gb=P, conv_w=P, A_log=P, dt_bias=P,
             gamma_o=P, W_o=P, S=P, conv_state=P, scale=128 ** -0.5, lower_bound=-5.0,
             rms_norm_eps=1e-5, l2_eps=1e-6, B=32, n=1, Hd=4096, nh=32, K=128, V=128, Kc=4,
             workspace=P, workspace_bytes=1 << 40, dev_status=None, stream=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,expect", [
    ({"B": -1}, ERR_SHAPE), ({"n": 0}, ERR_SHAPE), ({"Kc": 0}, ERR_SHAPE),
    ({"K": 64}, ERR_UNSUP), ({"Kc": 5}, ERR_UNSUP),
    ({"Hd": 4000}, ERR_UNSUP), ({"nh": 12}, ERR_UNSUP),
    ({"lower_bound": 1.0}, ERR_VALUE), ({"scale": float("inf")}, ERR_VALUE),
    ({"rms_norm_eps": -1.0}, ERR_VALUE),
    ({"W_in": None}, ERR_NULL), ({"S": None}, ERR_NULL),
    ({"W_o": P + 8}, ERR_ALIGN), ({"workspace": P + 16}, ERR_ALIGN),
    ({"workspace": None}, ERR_WS), ({"workspace_bytes": 1024}, ERR_WS),
    ({"B": 0}, KDA_OK),
])
def test_block_host_validation(lib, kw, expect):
    assert lib.kda_block_tkg(*block_args(**kw)) == expect


def test_block_workspace_size(lib):
    ws = lib.kda_block_tkg_workspace_size(32, 1, 4096, 32, 128, 128, 4)
    assert ws > 0 and ws % 256 == 0
    assert lib.kda_block_tkg_workspace_size(64, 1, 4096, 32, 128, 128, 4) > ws
    assert lib.kda_block_tkg_workspace_size(32, 2, 4096, 32, 128, 128, 4) > ws   # R = B * n rows
    assert lib.kda_block_tkg_workspace_size(32, 0, 4096, 32, 128, 128, 4) == 0
    assert lib.kda_block_tkg_workspace_size(32, 1, 4096, 12, 128, 128, 4) == 0


def decode_ex_args(**kw):
    a = dict(output=P, q=P, k=P, v=P, raw_gate=P, beta_logits=P, a_log=P, dt_bias=P,
             cu_seqlens=P, state_pool=P, state_indices=P, gate_mode=0, lower_bound=-5.0,
             state_layout=0, output_dtype=0, B=2, T=3, H=2, HV=4, K=128, V=128, max_slots=8,
             dev_status=None, stream=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,expect", [
    ({"state_layout": 2}, ERR_ENUM), ({"output_dtype": 2}, ERR_ENUM), ({"state_layout": -1}, ERR_ENUM),
    ({"output_dtype": 0, "output": P + 8}, ERR_ALIGN), ({"output_dtype": 1, "output": P + 4}, ERR_ALIGN),
    ({"B": 0, "state_layout": 1, "output_dtype": 1}, KDA_OK), ({"K": 64}, ERR_UNSUP),
])
def test_decode_ex_host_validation(lib, kw, expect):
    assert lib.kda_decode_ex(*decode_ex_args(**kw)) == expect


@pytest.mark.parametrize("kw,expect", [
    # gates the chunk form cannot take run the token-by-token kernel: their
    # calls validate like kda_decode's (here with no work to launch)
    ({"gate_mode": 0, "B": 0}, KDA_OK),
    ({"gate_mode": 1, "lower_bound": -6.0, "B": 0}, KDA_OK),
    ({"gate_mode": 2}, ERR_ENUM),
    ({"gate_mode": 1, "lower_bound": 0.5}, ERR_VALUE),
    ({"gate_mode": 1, "K": 64}, ERR_UNSUP),
    ({"gate_mode": 1, "B": 0}, KDA_OK),
])
def test_prefill_host_validation(lib, kw, expect):
    assert lib.kda_prefill(*decode_args(**kw)) == expect
