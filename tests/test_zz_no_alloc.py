"""kda_block_tkg_static: the block for callers that cannot allocate.

Such callers (a host whose memory pool owns every device allocation, a plugin
interface that only passes input and output buffers) cannot give the block a
workspace, so this entry point keeps its intermediates in a fixed array inside
the library.  These tests call it through the C ABI and check, on two calls in a row, that
it gives what kda_block_tkg with a caller workspace gives, within the parity
tolerances used everywhere else, and that the second call leaves the device's
free memory unchanged (nothing is allocated); that sizes beyond the fixed
array are refused; and that B = 0 and invalid sizes get the same status as
from kda_block_tkg without any CUDA call (so that check runs on a machine
without a GPU too).  The file is named to run after every other test file.
"""
import numpy as np
import pytest
import torch

from kda_decode_recurrence_gb300 import _lib, kda_block_tkg
from kda_decode_recurrence_gb300.inputs import block_inputs

from _parity import assert_outputs_close, assert_states_close, to_device

WEIGHTS = ("hidden", "gamma_in", "W_in", "W_fb", "W_gb", "conv_w", "A_log", "dt_bias",
           "gamma_o", "W_o")
KDA_ERR_WORKSPACE = -8


def call_static(inp, d, out, status):
    lib = _lib.load()
    return lib.kda_block_tkg_static(
        out.data_ptr(), *[d[k].data_ptr() for k in WEIGHTS], d["S"].data_ptr(),
        d["conv_state"].data_ptr(), inp["scale"], inp["lower_bound"], inp["rms_norm_eps"],
        inp["l2_eps"], inp["B"], inp["n"], inp["Hd"], inp["nh"], inp["K"], inp["V"], inp["Kc"],
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
@pytest.mark.parametrize("sizes", [{}, {"B": 5, "Hd": 256, "nh": 8, "seed": 81}],
                         ids=["kimi_k3_b32", "small"])
def test_static_scratch_matches_workspace_call_twice(sizes):
    inp = block_inputs(**sizes)
    ref = to_device(inp)      # advanced by kda_block_tkg with a caller workspace
    sta = to_device(inp)      # advanced by kda_block_tkg_static
    shape = (inp["B"], inp["n"], inp["Hd"])
    for call in range(2):     # the second call runs on the first call's leftovers
        out_ref = torch.full(shape, float("nan"), device="cuda")
        out_sta = torch.full(shape, float("nan"), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda_block_tkg(out_ref, *[ref[k] for k in WEIGHTS], ref["S"], ref["conv_state"],
                      inp["scale"], inp["lower_bound"], inp["rms_norm_eps"], inp["l2_eps"])
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert call_static(inp, sta, out_sta, status) == 0
        torch.cuda.synchronize()
        # The first call on a device may load the library's module (which
        # holds the fixed array); after that, no call allocates device memory.
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before
        assert status.item() == 0
        assert_outputs_close(out_sta.cpu().numpy(), out_ref.cpu().double().numpy(), "out")
        assert_states_close(sta["S"].cpu().numpy(), ref["S"].cpu().double().numpy(), "S")
        assert_outputs_close(sta["conv_state"].cpu().numpy(),
                             ref["conv_state"].cpu().double().numpy(), "conv_state")


@pytest.mark.gpu
def test_static_scratch_refuses_sizes_beyond_its_array():
    lib = _lib.load()
    need = lib.kda_block_tkg_workspace_size(4096, 1, 4096, 32, 128, 128, 4)
    assert need > 16 << 20
    fake = 0x10000   # never dereferenced: the size check comes first
    rc = lib.kda_block_tkg_static(*([fake] * 13), 128 ** -0.5, -5.0, 1e-5, 1e-6,
                                  4096, 1, 4096, 32, 128, 128, 4, None, None)
    assert rc == KDA_ERR_WORKSPACE


# B = 0 and sizes the block does not implement: both entry points must give
# the same status, before any CUDA call (the fake pointers are never used).
@pytest.mark.parametrize("B,n,Hd,nh,K,V,Kc", [
    (0, 1, 4096, 32, 128, 128, 4),      # no requests: KDA_OK
    (2, 1, 4096, 12, 128, 128, 4),      # num_head not a multiple of 8
    (2, 1, 4096, 32, 64, 64, 4),        # head dims other than 128
    (2, 0, 4096, 32, 128, 128, 4),      # n = 0
    (2, 1, 4000, 32, 128, 128, 4),      # Hd not a multiple of 128
    (-1, 1, 4096, 32, 128, 128, 4),     # negative B
])
def test_static_status_equals_workspace_call_without_cuda(B, n, Hd, nh, K, V, Kc):
    lib = _lib.load()
    fake = 0x10000
    ptrs, scalars, sizes = [fake] * 13, (128 ** -0.5, -5.0, 1e-5, 1e-6), (B, n, Hd, nh, K, V, Kc)
    rc_ws = lib.kda_block_tkg(*ptrs, *scalars, *sizes, None, 0, None, None)
    rc_static = lib.kda_block_tkg_static(*ptrs, *scalars, *sizes, None, None)
    assert rc_static == rc_ws
    assert (rc_ws == 0) == (B == 0)
