"""The decode and prefill kernels' timeout reports, exercised without a fault
or a hang.

Every wait of the decode kernel on a copy is bounded; when one gives up, the
CTA sets KDA_DEV_TIMEOUT, lets the copies it issued land (bounded again) and
returns, leaving its remaining work items unprocessed.  The test-only build
libkda_testhooks.so can withhold one work item's tile copy (its mbarrier phase
then never completes) and shorten the wait limit to 20 ms.  The CTA that owns
that item must report the timeout and skip its items; every other item must
be exactly as in a normal call; the context must stay usable.  The same build
can make one prefill (request, head) item's second MMA issuer skip the commit
of its first reads, so that the reads' barrier phase never completes: that
item must report the timeout and leave its outputs and state tile unwritten,
every other item must match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

from kda_decode_recurrence_gb300 import _lib
from kda_decode_recurrence_gb300.inputs import decode_inputs

from _parity import Guarded, assert_outputs_close, assert_states_close, guarded_copy, to_device

import oracle

pytestmark = pytest.mark.gpu

DEV_TIMEOUT = 4
FULL_WAIT_NS = 1_000_000_000


def hooks_lib():
    lib = _lib.load_variant("testhooks")
    lib.kda_test_set_decode_hooks.restype = None
    lib.kda_test_set_decode_hooks.argtypes = [ctypes.c_longlong, ctypes.c_ulonglong]
    return lib


def call(lib, inp, d, out, pool, status):
    return lib.kda_decode(out.data_ptr(), d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                          d["raw_gate"].data_ptr(), d["beta_logits"].data_ptr(),
                          d["a_log"].data_ptr(), d["dt_bias"].data_ptr(),
                          d["cu_seqlens"].data_ptr(), pool.data_ptr(),
                          d["state_indices"].data_ptr(), inp["gate_mode"], inp["lower_bound"],
                          inp["B"], inp["T"], inp["H"], inp["HV"], 128, 128, inp["max_slots"],
                          status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("tokens", [1, 2], ids=["single_token", "multi_token"])
def test_withheld_tile_copy_reports_timeout_and_spares_other_items(tokens):
    # one token per request: the single-token schedule; two: the multi-token one
    lib = hooks_lib()
    inp = decode_inputs("grouped", B=64, H=4, HV=8, max_slots=80, seed=140,
                        lengths=(tokens,) * 64)
    B, HV = inp["B"], inp["HV"]
    items = B * HV
    grid = min(items, 2 * torch.cuda.get_device_properties(0).multi_processor_count)
    withheld = 5
    # the CTA owning the withheld item fails on it and skips it and its later items
    if tokens == 1:
        skipped = set(range(withheld, items, grid))  # CTA c takes items c, c + G, ...
    else:
        # the multi-token kernel deals the items, ordered by request length
        # (all equal here, so by index), to the CTAs in a serpentine
        def owned(c):
            R, rem = divmod(items, grid)
            n = R + ((c < rem) if R % 2 == 0 else (grid - 1 - c < rem))
            return [j * grid + (c if j % 2 == 0 else grid - 1 - c) for j in range(n)]
        mine = next(owned(c) for c in range(grid) if withheld in owned(c))
        skipped = set(mine[mine.index(withheld):])
    d = to_device(inp)
    pool = guarded_copy(inp["state_pool"])
    out = Guarded((inp["T"], HV, 128), torch.float32, fill=float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_test_set_decode_hooks(withheld, 20_000_000)
    try:
        assert call(lib, inp, d, out.t, pool.t, status) == 0
        torch.cuda.synchronize()
    finally:
        lib.kda_test_set_decode_hooks(-1, FULL_WAIT_NS)
    assert out.intact() and pool.intact()
    assert status.item() == DEV_TIMEOUT
    ref_out, ref_pool, st = oracle.kda_decode(
        *[inp[k].double().numpy() for k in ("q", "k", "v", "raw_gate", "beta_logits", "a_log",
                                            "dt_bias")],
        inp["cu_seqlens"].numpy(), inp["state_pool"].double().numpy(),
        inp["state_indices"].numpy(), gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"])
    assert st == 0
    got_out, got_pool = out.t.cpu().numpy(), pool.t.cpu().numpy()
    idx = inp["state_indices"].numpy()
    before = inp["state_pool"].numpy()
    cu = inp["cu_seqlens"].numpy()
    for item in range(items):
        b, hv = divmod(item, HV)
        slot = idx[b]
        rows = slice(cu[b], cu[b + 1])
        if item in skipped:
            assert np.all(np.isnan(got_out[rows, hv]))                    # never written
            assert np.array_equal(got_pool[slot, hv], before[slot, hv])   # never stored
        else:
            assert_outputs_close(got_out[rows, hv], ref_out[rows, hv])
            assert_states_close(got_pool[slot, hv][None], ref_pool[slot, hv][None])
    # The context is still usable: the same call with no withheld item is complete.
    pool2 = guarded_copy(inp["state_pool"])
    out2 = Guarded((inp["T"], HV, 128), torch.float32, fill=float("nan"))
    status.zero_()
    assert call(lib, inp, d, out2.t, pool2.t, status) == 0
    torch.cuda.synchronize()
    assert status.item() == 0 and out2.intact() and pool2.intact()
    assert_outputs_close(out2.t.cpu().numpy(), ref_out)
    slots = torch.from_numpy(idx.astype(np.int64))
    assert_states_close(pool2.t.cpu()[slots].numpy(), ref_pool[idx])


def test_prefill_uncommitted_reads_report_timeout_and_spare_other_items():
    lib = _lib.load_variant("testhooks")
    lib.kda_test_set_prefill_hooks.restype = None
    lib.kda_test_set_prefill_hooks.argtypes = [ctypes.c_longlong, ctypes.c_ulonglong]
    inp = decode_inputs("varlen", B=4, H=4, HV=8, max_slots=6, seed=141, lengths=(40, 17, 33, 16))
    assert inp["gate_mode"] == 1 and inp["lower_bound"] >= -5.0  # the chunk form runs
    B, HV = inp["B"], inp["HV"]
    withheld = 5                                                 # request 0, head 5
    d = to_device(inp)
    pool = guarded_copy(inp["state_pool"])
    out = Guarded((inp["T"], HV, 128), torch.float32, fill=float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(o, pl):
        return lib.kda_prefill(o.data_ptr(), d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                               d["raw_gate"].data_ptr(), d["beta_logits"].data_ptr(),
                               d["a_log"].data_ptr(), d["dt_bias"].data_ptr(),
                               d["cu_seqlens"].data_ptr(), pl.data_ptr(),
                               d["state_indices"].data_ptr(), inp["gate_mode"], inp["lower_bound"],
                               B, inp["T"], inp["H"], HV, 128, 128, inp["max_slots"],
                               status.data_ptr(), torch.cuda.current_stream().cuda_stream)

    lib.kda_test_set_prefill_hooks(withheld, 20_000_000)
    try:
        assert run(out.t, pool.t) == 0
        torch.cuda.synchronize()
    finally:
        lib.kda_test_set_prefill_hooks(-1, FULL_WAIT_NS)
    assert out.intact() and pool.intact()
    assert status.item() == DEV_TIMEOUT
    ref_out, ref_pool, st = oracle.kda_decode(
        *[inp[k].double().numpy() for k in ("q", "k", "v", "raw_gate", "beta_logits", "a_log",
                                            "dt_bias")],
        inp["cu_seqlens"].numpy(), inp["state_pool"].double().numpy(),
        inp["state_indices"].numpy(), gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"])
    assert st == 0
    got_out, got_pool = out.t.cpu().numpy(), pool.t.cpu().numpy()
    idx = inp["state_indices"].numpy()
    before = inp["state_pool"].numpy()
    cu = inp["cu_seqlens"].numpy()
    for item in range(B * HV):
        b, hv = divmod(item, HV)
        rows = slice(cu[b], cu[b + 1])
        if item == withheld:
            assert np.all(np.isnan(got_out[rows, hv]))
            assert np.array_equal(got_pool[idx[b], hv], before[idx[b], hv])
        else:
            assert_outputs_close(got_out[rows, hv], ref_out[rows, hv])
            assert_states_close(got_pool[idx[b], hv][None], ref_pool[idx[b], hv][None])
    # The context is still usable: the same call with nothing withheld is complete.
    pool2 = guarded_copy(inp["state_pool"])
    out2 = Guarded((inp["T"], HV, 128), torch.float32, fill=float("nan"))
    status.zero_()
    assert run(out2.t, pool2.t) == 0
    torch.cuda.synchronize()
    assert status.item() == 0 and out2.intact() and pool2.intact()
    assert_outputs_close(out2.t.cpu().numpy(), ref_out)
    slots = torch.from_numpy(idx.astype(np.int64))
    assert_states_close(pool2.t.cpu()[slots].numpy(), ref_pool[idx])
