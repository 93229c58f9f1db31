"""GB300-native KDA token-generation library: Python binding of libkda.

The functions are the C-ABI calls of include/kda.h, under the same names;
this module only checks tensors and marshals their device pointers, sizes and
the current CUDA stream.  Every step of the computation runs in libkda's CUDA
kernels; there is no CPU or PyTorch fallback, and a missing library raises.

Each call returns its device status word (an int32 CUDA tensor: KDA_DEV_*
bits the kernels OR in).  Pass ``dev_status`` to reuse one; when none is
passed, a zeroed word is allocated on the call's stream, so that device-side
reports (a bad slot, a malformed cu_seqlens, a pipeline timeout) are never
dropped.  ``check_device=True`` synchronises the stream and raises
KdaDeviceError when any bit is set.

    kda_decode(output, q, k, v, raw_gate, beta_logits, a_log, dt_bias,
               cu_seqlens, state_pool, state_indices, gate_mode, lower_bound)
    kda_decode_ex(..., state_layout=STATE_K_FIRST | STATE_V_FIRST)
               (the output dtype, fp32 or bf16, is taken from `output`)
    kda_prefill(<the arguments of kda_decode>)   16-token chunks
    kda_block_tkg(out, hidden, gamma_in, W_in, W_fb, W_gb, conv_w, A_log,
                  dt_bias, gamma_o, W_o, S, conv_state, scale, lower_bound,
                  rms_norm_eps, l2_eps, workspace)
    block_workspace_size(B, n, Hd, nh, K, V, Kc)
"""
from __future__ import annotations

import torch

from . import _lib

GATE_SOFTPLUS = 0
GATE_LOWER_BOUND = 1
STATE_K_FIRST = 0
STATE_V_FIRST = 1
OUTPUT_F32 = 0
OUTPUT_BF16 = 1
DEV_BAD_SLOT = 1
DEV_BAD_SEQLEN = 2
DEV_TIMEOUT = 4
DEV_BOUNDS = 8  # debug builds only (libkda_debugbounds.so)


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = _lib.STATUS.get(status, str(status))
        super().__init__(f"{what} failed: {name} ({_lib.load().kda_status_string(status).decode()})")


class KdaDeviceError(RuntimeError):
    def __init__(self, bits: int, what: str):
        self.bits = bits
        names = [n for b, n in ((DEV_BAD_SLOT, "KDA_DEV_BAD_SLOT"),
                                (DEV_BAD_SEQLEN, "KDA_DEV_BAD_SEQLEN"),
                                (DEV_TIMEOUT, "KDA_DEV_TIMEOUT"),
                                (DEV_BOUNDS, "KDA_DEV_BOUNDS")) if bits & b]
        super().__init__(f"{what}: device status {bits} ({' | '.join(names) or 'unknown bits'})")


def _check(t: torch.Tensor, name: str, dtype, device) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _status_word(dev_status, device, stream) -> torch.Tensor:
    """The caller's status word, or a new zeroed one, ordered on the call's
    stream (so the zeroing precedes the kernels that OR into it)."""
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, device)
        return dev_status
    with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream(device)):
        return torch.zeros(1, dtype=torch.int32, device=device)


def _finish(rc: int, status: torch.Tensor, what: str, check: bool, check_device: bool, stream):
    if check and rc != 0:
        raise KdaError(rc, what)
    if check_device and rc == 0:
        (stream if stream is not None else torch.cuda.current_stream(status.device)).synchronize()
        bits = int(status.item())
        if bits != 0:
            raise KdaDeviceError(bits, what)
    return status


def kda_decode(output, q, k, v, raw_gate, beta_logits, a_log, dt_bias, cu_seqlens, state_pool,
               state_indices, gate_mode=GATE_SOFTPLUS, lower_bound=-5.0, dev_status=None,
               stream=None, check=True, check_device=False) -> torch.Tensor:
    """Advance the slot-indexed states over the packed tokens (see include/kda.h).

    Shapes (a leading batch axis of 1 is accepted): output [T, HV, V] fp32;
    q, k [T, H, K] bf16; v [T, HV, V] bf16; raw_gate [T, HV, K] fp32;
    beta_logits [T, HV] fp32; a_log [HV] fp32; dt_bias [HV, K] fp32;
    cu_seqlens [B+1] int32; state_pool [N, HV, K, V] fp32 (advanced in place);
    state_indices [B] int32.  Returns the device status word; raises KdaError
    on a negative C status when ``check`` (see the module docstring for
    ``dev_status`` and ``check_device``).
    """
    dev = state_pool.device
    T = q.shape[-3]
    H, K = q.shape[-2], q.shape[-1]
    HV, V = v.shape[-2], v.shape[-1]
    B = state_indices.shape[0]
    N = state_pool.shape[0]
    for t, n, dt in ((output, "output", torch.float32), (q, "q", torch.bfloat16),
                     (k, "k", torch.bfloat16), (v, "v", torch.bfloat16),
                     (raw_gate, "raw_gate", torch.float32),
                     (beta_logits, "beta_logits", torch.float32), (a_log, "a_log", torch.float32),
                     (dt_bias, "dt_bias", torch.float32), (cu_seqlens, "cu_seqlens", torch.int32),
                     (state_pool, "state_pool", torch.float32),
                     (state_indices, "state_indices", torch.int32)):
        _check(t, n, dt, dev)
    if tuple(state_pool.shape[1:]) != (HV, K, V):
        raise ValueError(f"state_pool shape {tuple(state_pool.shape)} != [N, {HV}, {K}, {V}]")
    if cu_seqlens.numel() != B + 1:
        raise ValueError("cu_seqlens must have B + 1 entries")
    status = _status_word(dev_status, dev, stream)
    rc = _lib.load().kda_decode(
        output.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), raw_gate.data_ptr(),
        beta_logits.data_ptr(), a_log.data_ptr(), dt_bias.data_ptr(), cu_seqlens.data_ptr(),
        state_pool.data_ptr(), state_indices.data_ptr(), int(gate_mode), float(lower_bound),
        B, T, H, HV, K, V, N, status.data_ptr(), _stream_handle(stream))
    return _finish(rc, status, "kda_decode", check, check_device, stream)


def kda_prefill(output, q, k, v, raw_gate, beta_logits, a_log, dt_bias, cu_seqlens, state_pool,
                state_indices, gate_mode=GATE_LOWER_BOUND, lower_bound=-5.0, dev_status=None,
                stream=None, check=True, check_device=False) -> torch.Tensor:
    """Whole-prompt prefill: the kda_decode recurrence computed 16 tokens at a
    time for the lower-bound gate with lower_bound >= -5; other gates run the
    token-by-token kernel.  Same tensors as kda_decode."""
    dev = state_pool.device
    T = q.shape[-3]
    H, K = q.shape[-2], q.shape[-1]
    HV, V = v.shape[-2], v.shape[-1]
    B = state_indices.shape[0]
    N = state_pool.shape[0]
    for t, n, dt in ((output, "output", torch.float32), (q, "q", torch.bfloat16),
                     (k, "k", torch.bfloat16), (v, "v", torch.bfloat16),
                     (raw_gate, "raw_gate", torch.float32),
                     (beta_logits, "beta_logits", torch.float32), (a_log, "a_log", torch.float32),
                     (dt_bias, "dt_bias", torch.float32), (cu_seqlens, "cu_seqlens", torch.int32),
                     (state_pool, "state_pool", torch.float32),
                     (state_indices, "state_indices", torch.int32)):
        _check(t, n, dt, dev)
    if tuple(state_pool.shape[1:]) != (HV, K, V):
        raise ValueError(f"state_pool shape {tuple(state_pool.shape)} != [N, {HV}, {K}, {V}]")
    if cu_seqlens.numel() != B + 1:
        raise ValueError("cu_seqlens must have B + 1 entries")
    status = _status_word(dev_status, dev, stream)
    rc = _lib.load().kda_prefill(
        output.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), raw_gate.data_ptr(),
        beta_logits.data_ptr(), a_log.data_ptr(), dt_bias.data_ptr(), cu_seqlens.data_ptr(),
        state_pool.data_ptr(), state_indices.data_ptr(), int(gate_mode), float(lower_bound),
        B, T, H, HV, K, V, N, status.data_ptr(), _stream_handle(stream))
    return _finish(rc, status, "kda_prefill", check, check_device, stream)


def kda_decode_ex(output, q, k, v, raw_gate, beta_logits, a_log, dt_bias, cu_seqlens, state_pool,
                  state_indices, gate_mode=GATE_SOFTPLUS, lower_bound=-5.0,
                  state_layout=STATE_K_FIRST, dev_status=None, stream=None, check=True,
                  check_device=False) -> torch.Tensor:
    """kda_decode with a chosen state layout (STATE_K_FIRST: tiles [K, V];
    STATE_V_FIRST: tiles [V, K]) and the output dtype taken from ``output``
    (float32 or bfloat16)."""
    dev = state_pool.device
    T = q.shape[-3]
    H, K = q.shape[-2], q.shape[-1]
    HV, V = v.shape[-2], v.shape[-1]
    B = state_indices.shape[0]
    N = state_pool.shape[0]
    if output.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"output: expected float32 or bfloat16, got {output.dtype}")
    out_dtype = OUTPUT_F32 if output.dtype == torch.float32 else OUTPUT_BF16
    _check(output, "output", output.dtype, dev)
    for t, n, dt in ((q, "q", torch.bfloat16), (k, "k", torch.bfloat16), (v, "v", torch.bfloat16),
                     (raw_gate, "raw_gate", torch.float32),
                     (beta_logits, "beta_logits", torch.float32), (a_log, "a_log", torch.float32),
                     (dt_bias, "dt_bias", torch.float32), (cu_seqlens, "cu_seqlens", torch.int32),
                     (state_pool, "state_pool", torch.float32),
                     (state_indices, "state_indices", torch.int32)):
        _check(t, n, dt, dev)
    tile = (K, V) if state_layout == STATE_K_FIRST else (V, K)
    if tuple(state_pool.shape[1:]) != (HV, *tile):
        raise ValueError(f"state_pool shape {tuple(state_pool.shape)} != [N, {HV}, {tile[0]}, {tile[1]}]")
    if cu_seqlens.numel() != B + 1:
        raise ValueError("cu_seqlens must have B + 1 entries")
    status = _status_word(dev_status, dev, stream)
    rc = _lib.load().kda_decode_ex(
        output.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), raw_gate.data_ptr(),
        beta_logits.data_ptr(), a_log.data_ptr(), dt_bias.data_ptr(), cu_seqlens.data_ptr(),
        state_pool.data_ptr(), state_indices.data_ptr(), int(gate_mode), float(lower_bound),
        int(state_layout), out_dtype, B, T, H, HV, K, V, N,
        status.data_ptr(), _stream_handle(stream))
    return _finish(rc, status, "kda_decode_ex", check, check_device, stream)


def block_workspace_size(B, n, Hd, nh, K, V, Kc) -> int:
    return int(_lib.load().kda_block_tkg_workspace_size(B, n, Hd, nh, K, V, Kc))


def kda_block_tkg(out, hidden, gamma_in, W_in, W_fb, W_gb, conv_w, A_log, dt_bias, gamma_o, W_o,
                  S, conv_state, scale, lower_bound, rms_norm_eps=1e-5, l2_eps=1e-6,
                  workspace=None, dev_status=None, stream=None, check=True,
                  check_device=False) -> torch.Tensor:
    """The fused KDA block (see include/kda.h).  ``workspace`` is a uint8 CUDA
    tensor of at least block_workspace_size(...) bytes; when None one is
    allocated here with torch (device memory plumbing only)."""
    dev = hidden.device
    B, n, Hd = hidden.shape
    _, nh, K, V = S.shape
    Kc = conv_state.shape[-1] + 1
    for t, name, dt in ((out, "out", torch.float32), (hidden, "hidden", torch.float32),
                        (gamma_in, "gamma_in", torch.float32), (W_in, "W_in", torch.bfloat16),
                        (W_fb, "W_fb", torch.bfloat16), (W_gb, "W_gb", torch.bfloat16),
                        (conv_w, "conv_w", torch.bfloat16), (A_log, "A_log", torch.float32),
                        (dt_bias, "dt_bias", torch.float32), (gamma_o, "gamma_o", torch.float32),
                        (W_o, "W_o", torch.bfloat16), (S, "S", torch.float32),
                        (conv_state, "conv_state", torch.float32)):
        _check(t, name, dt, dev)
    need = block_workspace_size(B, n, Hd, nh, K, V, Kc)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    status = _status_word(dev_status, dev, stream)
    rc = _lib.load().kda_block_tkg(
        out.data_ptr(), hidden.data_ptr(), gamma_in.data_ptr(), W_in.data_ptr(), W_fb.data_ptr(),
        W_gb.data_ptr(), conv_w.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr(),
        gamma_o.data_ptr(), W_o.data_ptr(), S.data_ptr(), conv_state.data_ptr(), float(scale),
        float(lower_bound), float(rms_norm_eps), float(l2_eps), B, n, Hd, nh, K, V, Kc,
        workspace.data_ptr(), workspace.numel(), status.data_ptr(), _stream_handle(stream))
    return _finish(rc, status, "kda_block_tkg", check, check_device, stream)


def version() -> str:
    return _lib.load().kda_version().decode()
