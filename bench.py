#!/usr/bin/env python
"""Benchmark: KDA decode state-updates/s and HBM roofline fraction on GB300.

One step = one kda_decode call (C ABI) over the large-batch grouped decode
workload: B = 256 requests x 1 token, key heads H = 48, value heads HV = 96
(G = 2), dk = dv = 128, state pool [512, 96, 128, 128] fp32 (3.2 GB, far
larger than L2, so no flush is needed between steps), softplus gate.  The
state pool is advanced in place step after step (bounded: beta <= 1, unit
keys, exp(g) <= 1).

Printed (rank 0, one JSON line): state-updates/s (req x head x token), the
decode kernel's roofline against the measured HBM copy bandwidth, an
end-to-end figure through host buffers, SM clocks sampled during the timed
region, the float64 oracle timed on the host cores, and the fused block
(kda_block_tkg, B = 32, Hd = 4096, nh = 32) timed separately.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kda_decode_recurrence_gb300.inputs import (BLOCK_CONFIG, DECODE_CONFIGS,  # noqa: E402
                                                block_inputs, decode_inputs, to_f64)

METRIC = "KDA decode state-updates/s (req·head·token) and HBM GB/s vs GB300 peak"
UNIT = "state-updates/s"
WORKLOAD = "grouped"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per launch of the decode kernel, tied to the kernel sources they
# were taken with (when the sources change the figure no longer describes the
# kernel and is reported as null).  Taken by ncu on the reduced case (B = 32
# requests, one eighth of the grouped workload: `bench.py --profile decode`)
# and scaled to the full launch: reads x 8; writes x 8 less what is still
# dirty in L2 when the kernel ends (the reduced case's algorithmic writes
# minus its measured ones, 55.2 MB), which does not grow with the workload.
NCU_REDUCED = {"read": 204660992, "write": 147660544, "algorithmic_write": 202899456, "scale": 8}
NCU_TRAFFIC = {"sources_sha256": "ad45e14dfdb5a47ad6fe947108b664dbad52393d5635ff7dbb9604994e466120",
               "bytes_per_launch": (NCU_REDUCED["read"] * NCU_REDUCED["scale"]
                                    + NCU_REDUCED["algorithmic_write"] * NCU_REDUCED["scale"]
                                    - (NCU_REDUCED["algorithmic_write"] - NCU_REDUCED["write"]))}


def kernel_sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kda_decode_recurrence_gb300", "csrc")
    for f in ("kda_common.cuh", "kda_async.cuh", "kda_recurrence.cuh", "kda_decode.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def decode_bytes(B, T, H, HV, K, V, touched=None) -> int:
    """Algorithmic HBM bytes of one kda_decode call: each advanced state tile
    read and written once, q/k once per key head (bf16), v (bf16), raw_gate,
    beta_logits, output (fp32), a_log, dt_bias, cu_seqlens, state_indices."""
    touched = B if touched is None else touched
    return (touched * HV * 2 * K * V * 4
            + T * (H * K * 2 * 2 + HV * V * 2 + HV * K * 4 + HV * 4 + HV * V * 4)
            + HV * (K + 1) * 4 + (2 * B + 1) * 4)


def block_bytes(B, Hd, nh, K, V, Kc, n=1) -> int:
    """Algorithmic HBM bytes of one kda_block_tkg call: weights once, S and
    conv_state read + written, hidden in and out out for the B * n tokens,
    small parameters."""
    I = 2 * K * nh + V * nh + 2 * K + nh
    weights = 2 * (Hd * I + K * K * nh + K * V * nh + 3 * Kc * K * nh + V * nh * Hd)
    params = 4 * (Hd + nh + K * nh + V)
    state = B * nh * K * V * 4 * 2 + B * 3 * K * nh * (Kc - 1) * 4 * 2
    io = B * n * Hd * 4 * 2
    return weights + params + state + io


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    QUERY = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not inside and self.samples:  # region shorter than one sample period
            nearest = min(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))
            inside = [nearest[1]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside)}


def device_uuid():
    try:
        u = str(torch.cuda.get_device_properties(0).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: the job's time."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch (own requests, own pool slots): weak scaling."""
    return base_seed + 1000 * rank


# ----------------------------------------------------------------- oracle


def cpu_info() -> dict:
    """The host CPU: model name (lscpu, else /proc/cpuinfo), logical CPUs,
    and the cores this process may use."""
    from oracle.parallel import host_cores
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            fields = {}
            for line in open("/proc/cpuinfo"):
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
            model = fields.get("model name") or (
                f"implementer {fields.get('CPU implementer')} part {fields.get('CPU part')}"
                if "CPU part" in fields else None)
        except Exception:
            pass
    import platform
    return {"cpu_model": model or platform.machine(), "nproc": os.cpu_count(),
            "cores_usable": host_cores()}


def decode_oracle_arrays(inp: dict) -> tuple:
    """A decode workload as the oracle workers read it: tokens (bf16 values
    widened exactly to fp32), and the requests' state tiles in request order.
    Returns (arrays, (gate_mode, lower_bound), state updates)."""
    from oracle import parallel as P
    idx = inp["state_indices"].long()
    tok = {k: inp[k].float().numpy() for k in P.DECODE_TOKENS}
    arrays = P.decode_arrays(tok, inp["a_log"].numpy(), inp["dt_bias"].numpy(),
                             inp["cu_seqlens"].numpy(), inp["state_pool"][idx].numpy())
    return arrays, (inp["gate_mode"], inp["lower_bound"]), inp["T"] * inp["HV"]


def cpu_baseline(main_inp: dict) -> dict:
    """The float64 oracle, as it stands, on this host: every workload (the
    four decode ones and the block) in full, once on one thread and once
    split by request over all usable cores (one spawned worker process per
    core).  The headline value is the all-cores rate on the bench workload."""
    from oracle import parallel as P
    info = cpu_info()
    cores = info["cores_usable"]
    per = {}
    with P.OracleWorkers(cores) as w:
        for name in ("tiny", "single", "grouped", "varlen"):
            inp = main_inp if name == WORKLOAD else decode_inputs(name)
            arrays, extra, upd = decode_oracle_arrays(inp)
            B = inp["B"]
            del inp
            t1 = P.time_single("decode", arrays, B, extra)
            staged = w.stage(arrays)
            del arrays
            tn = min(w.run("decode", staged, B, extra) for _ in range(2))
            per[name] = {"state_updates": upd, "single_thread": upd / t1, "all_cores": upd / tn,
                         "seconds_single": t1, "seconds_all_cores": tn}
        binp = block_inputs()
        params = {k: binp[k].float().numpy() for k in P.BLOCK_WEIGHTS}
        arrays = P.block_arrays(params, binp["hidden"].numpy(), binp["S"].numpy(),
                                binp["conv_state"].numpy())
        extra = (binp["scale"], binp["lower_bound"], binp["rms_norm_eps"], binp["l2_eps"])
        upd = binp["B"] * binp["n"] * binp["nh"]
        t1 = P.time_single("block", arrays, binp["B"], extra)
        staged = w.stage(arrays)
        tn = min(w.run("block", staged, binp["B"], extra) for _ in range(2))
        per["block"] = {"state_updates": upd, "single_thread": upd / t1, "all_cores": upd / tn,
                        "seconds_single": t1, "seconds_all_cores": tn}
    main = per[WORKLOAD]
    return {"value": main["all_cores"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"whole workloads: every request of {WORKLOAD} (B={main_inp['B']}, "
                       f"{main['state_updates']} state updates) and of tiny, single, varlen and "
                       "block; float64 C oracle, split by request over one spawned process per "
                       "core (best of 2 passes), and on one thread"),
            "single_thread": {"value": main["single_thread"], "cores": 1},
            "cpu_model": info["cpu_model"], "nproc": info["nproc"], "per_workload": per}


def config_dict(cfg) -> dict:
    return {"workload": f"{cfg.name} decode: B={cfg.B} x 1 token, H={cfg.H}, HV={cfg.HV} "
                        f"(G={cfg.HV // cfg.H}), dk=dv={cfg.K}, state_pool [{cfg.max_slots}, {cfg.HV}, "
                        f"{cfg.K}, {cfg.V}] fp32, softplus gate",
            "B": cfg.B, "T": cfg.B, "H": cfg.H, "HV": cfg.HV, "K": cfg.K, "V": cfg.V,
            "max_slots": cfg.max_slots, "gate_mode": "softplus", "seed": cfg.seed,
            "l2": "no flush: the 3.2 GB state pool is larger than L2 (129 MB)"}


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle on the host cores.  Each step is
    one pass over every request of the bench workload, split by request over
    one spawned worker process per usable core."""
    if rank != 0:
        return
    from oracle import parallel as P
    cfg = DECODE_CONFIGS[WORKLOAD]
    inp = decode_inputs(cfg)
    arrays, extra, upd = decode_oracle_arrays(inp)
    B = inp["B"]
    del inp
    info = cpu_info()
    cores = info["cores_usable"]
    with P.OracleWorkers(cores) as w:
        staged = w.stage(arrays)
        del arrays
        for _ in range(args.warmup):
            w.run("decode", staged, B, extra)
        times = [w.run("decode", staged, B, extra) for _ in range(args.steps)]
    elapsed = sum(times)
    value = upd * args.steps / elapsed
    sample = (f"each step: all {B} requests x {cfg.HV} value heads ({upd} state updates), "
              f"float64 C oracle split by request over {cores} worker processes "
              f"({info['cpu_model']}, {info['nproc']} logical CPUs)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu_model": info["cpu_model"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU arm


def run_block(steps: int, warmup: int, n: int = 1) -> dict:
    from kda_decode_recurrence_gb300 import block_workspace_size, kda_block_tkg
    cfg = BLOCK_CONFIG
    inp = block_inputs(cfg, n=n)
    dev = "cuda"
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty(cfg.B, n, cfg.Hd, device=dev)
    ws = torch.empty(block_workspace_size(cfg.B, n, cfg.Hd, cfg.nh, cfg.K, cfg.V, cfg.Kc),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    names = ("hidden", "gamma_in", "W_in", "W_fb", "W_gb", "conv_w", "A_log", "dt_bias",
             "gamma_o", "W_o")

    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        kda_block_tkg(out, *[d[k] for k in names], d["S"], d["conv_state"], inp["scale"],
                      inp["lower_bound"], inp["rms_norm_eps"], inp["l2_eps"], workspace=ws,
                      dev_status=status)

    for _ in range(warmup):
        call()
    stream = torch.cuda.current_stream()

    def timed(fn, flush_l2=True):
        times = []
        for _ in range(steps):
            if flush_l2:
                flush.fill_(1)  # evict L2 between calls
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            e.synchronize()
            times.append(s.elapsed_time(e) * 1e-3)
        return statistics.median(times)

    t_eager = timed(call)
    # The same call captured once in a CUDA graph and replayed: the device time
    # of the kernel chain without the host's per-launch work in between.
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        call()
    stream.wait_stream(side)
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        call()
    t = timed(graph.replay)
    # Hot cache: the same replay back to back, without the flush (the weights
    # and part of S may still be in the 129 MB L2 from the previous call).
    t_hot = timed(graph.replay, flush_l2=False)
    nbytes = block_bytes(cfg.B, cfg.Hd, cfg.nh, cfg.K, cfg.V, cfg.Kc, n)
    peak, src = measured_peaks()
    return {"workload": f"kda_block_tkg B={cfg.B} n={n} Hd={cfg.Hd} nh={cfg.nh} dk=dv={cfg.K} "
                        f"Kc={cfg.Kc}, L2 flushed before each call",
            "us_per_call": t * 1e6, "us_per_call_eager": t_eager * 1e6,
            "us_per_call_hot_l2": t_hot * 1e6,
            "timing": "CUDA graph replay of one C-ABI call (eager: host launches each call)",
            "calls": steps, "gpu_launches_per_call": 6,
            "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / t / 1e9,
            "frac_of_hbm_peak": nbytes / t / 1e9 / peak, "peak_source": src,
            "state_updates_per_s": cfg.B * n * cfg.nh / t}


def run_block_eager(steps: int, warmup: int, n: int = 1) -> dict:
    """The block as eager C-ABI calls only (no CUDA graph), L2 flushed before
    each: the case for kernel-level ncu captures, which cannot replay the
    nodes of a captured graph with programmatic-dependency edges."""
    from kda_decode_recurrence_gb300 import block_workspace_size, kda_block_tkg
    cfg = BLOCK_CONFIG
    inp = block_inputs(cfg, n=n)
    d = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty(cfg.B, n, cfg.Hd, device="cuda")
    ws = torch.empty(block_workspace_size(cfg.B, n, cfg.Hd, cfg.nh, cfg.K, cfg.V, cfg.Kc),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    names = ("hidden", "gamma_in", "W_in", "W_fb", "W_gb", "conv_w", "A_log", "dt_bias",
             "gamma_o", "W_o")
    times = []
    for i in range(warmup + steps):
        flush.fill_(1)
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record()
        kda_block_tkg(out, *[d[k] for k in names], d["S"], d["conv_state"], inp["scale"],
                      inp["lower_bound"], inp["rms_norm_eps"], inp["l2_eps"], workspace=ws,
                      dev_status=status)
        e_.record()
        e_.synchronize()
        if i >= warmup:
            times.append(s_.elapsed_time(e_) * 1e-3)
    assert status.item() == 0
    return {"workload": f"kda_block_tkg B={cfg.B} n={n}, eager calls, L2 flushed before each",
            "us_per_call": statistics.median(times) * 1e6, "calls": steps}


def run_decode_variant(inp: dict, d: dict, steps: int) -> dict:
    """kda_decode_ex on the same workload with the transposed (V-first) state
    and bf16 output, timed like the main step (CUDA events per launch)."""
    from kda_decode_recurrence_gb300 import STATE_V_FIRST, kda_decode_ex
    T, H, HV, K, V, B = inp["T"], inp["H"], inp["HV"], inp["K"], inp["V"], inp["B"]
    pool = d["state_pool"].transpose(-1, -2).contiguous()
    out = torch.empty(T, HV, V, dtype=torch.bfloat16, device=pool.device)
    stream = torch.cuda.current_stream(pool.device)
    status = torch.zeros(1, dtype=torch.int32, device=pool.device)

    def call():
        kda_decode_ex(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
                      d["dt_bias"], d["cu_seqlens"], pool, d["state_indices"],
                      gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"],
                      state_layout=STATE_V_FIRST, dev_status=status, stream=stream)

    for _ in range(3):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s_, e_ in ev:
        s_.record(stream)
        call()
        e_.record(stream)
    torch.cuda.synchronize(pool.device)
    t = sum(s_.elapsed_time(e_) for s_, e_ in ev) * 1e-3 / steps
    nbytes = decode_bytes(B, T, H, HV, K, V) - T * HV * V * 2   # bf16 output
    peak, src = measured_peaks()
    del pool
    return {"workload": "same as config, state_layout V_FIRST ([V, K] tiles), bf16 output",
            "us_per_launch": t * 1e6, "launches": steps, "algorithmic_bytes": nbytes,
            "achieved_gbs": nbytes / t / 1e9, "frac_of_hbm_peak": nbytes / t / 1e9 / peak,
            "peak_source": src, "state_updates_per_s": T * HV / t}


def run_decode_varlen(steps: int) -> dict:
    """kda_decode on the varlen workload (64 requests of 1..8 tokens, H = HV =
    96, lower-bound gate): the kernel's multi-token path, where each state
    tile carries several tokens.  CUDA events per launch; the 805 MB pool is
    far above L2."""
    from kda_decode_recurrence_gb300 import kda_decode
    inp = decode_inputs(DECODE_CONFIGS["varlen"])
    dev = torch.device("cuda", torch.cuda.current_device())
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    T, H, HV, K, V, B = inp["T"], inp["H"], inp["HV"], inp["K"], inp["V"], inp["B"]
    out = torch.empty(T, HV, V, device=dev)
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        kda_decode(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
                   d["dt_bias"], d["cu_seqlens"], d["state_pool"], d["state_indices"],
                   gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"],
                   dev_status=status, stream=stream)

    for _ in range(3):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s_, e_ in ev:
        s_.record(stream)
        call()
        e_.record(stream)
    torch.cuda.synchronize(dev)
    t = sum(s_.elapsed_time(e_) for s_, e_ in ev) * 1e-3 / steps
    nbytes = decode_bytes(B, T, H, HV, K, V)
    peak, src = measured_peaks()
    return {"workload": f"varlen decode: B={B} requests of 1..8 tokens (T={T}), H=HV={HV}, "
                        f"dk=dv={K}, pool [{inp['state_pool'].shape[0]}, {HV}, {K}, {V}] fp32, "
                        "lower-bound gate -5",
            "us_per_launch": t * 1e6, "launches": steps, "algorithmic_bytes": nbytes,
            "achieved_gbs": nbytes / t / 1e9, "frac_of_hbm_peak": nbytes / t / 1e9 / peak,
            "peak_source": src, "state_updates_per_s": T * HV / t}


def prefill_flops(T: int, HV: int, K: int, V: int) -> int:
    """fp32 flops of the recurrence over T tokens of HV heads: per token and
    head the decay (K*V), k^T S (2 K V), the rank-1 write (2 K V) and the read
    (2 K V)."""
    return T * HV * 7 * K * V


def run_prefill(steps: int, warmup: int) -> dict:
    """Whole-prompt prefill: B = 2 requests x 2048 tokens, H = HV = 96,
    lower-bound gate, state from the pool, final state written back; timed
    for the chunked kda_prefill and for kda_decode's token-by-token kernel."""
    res = {"chunked": _prefill_once(steps, warmup, "chunked"),
           "recurrent": _prefill_once(steps, warmup, "recurrent")}
    res["speedup_chunked_vs_recurrent"] = res["recurrent"]["ms"] / res["chunked"]["ms"]
    return res


def _prefill_once(steps: int, warmup: int, impl: str) -> dict:
    from kda_decode_recurrence_gb300 import kda_decode, kda_prefill
    fn = kda_prefill if impl == "chunked" else kda_decode
    B, L = 2, 2048
    inp = decode_inputs(DECODE_CONFIGS["varlen"], B=B, H=96, HV=96, max_slots=4,
                        lengths=(L,) * B, seed=7)
    dev = torch.device("cuda", 0)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty(inp["T"], inp["HV"], inp["V"], device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        fn(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
           d["dt_bias"], d["cu_seqlens"], d["state_pool"], d["state_indices"],
           gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"], dev_status=status)

    for _ in range(warmup):
        call()
    times = []
    for _ in range(steps):
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record()
        call()
        e_.record()
        e_.synchronize()
        times.append(s_.elapsed_time(e_) * 1e-3)
    t = statistics.median(times)
    fl = prefill_flops(inp["T"], inp["HV"], inp["K"], inp["V"])
    return {"impl": impl, "workload": f"prefill B={B} x {L} tokens, H=HV=96, lower-bound gate",
            "ms": t * 1e3, "tokens_per_s": inp["T"] / t, "state_updates_per_s": inp["T"] * inp["HV"] / t,
            "tflops": fl / t / 1e12}


def run_gpu(args, rank, world, local):
    from kda_decode_recurrence_gb300 import kda_decode
    cfg = DECODE_CONFIGS[WORKLOAD]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = decode_inputs(cfg, seed=shard_seed(cfg.seed, rank))
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    B, T, H, HV, K, V = inp["B"], inp["T"], inp["H"], inp["HV"], inp["K"], inp["V"]
    out = torch.empty(T, HV, V, device=dev)
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        kda_decode(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
                   d["dt_bias"], d["cu_seqlens"], d["state_pool"], d["state_indices"],
                   gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"],
                   dev_status=status, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(device_uuid())
    sampler.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    w0 = time.time()
    for s, e in ev:
        s.record(stream)
        step()
        e.record(stream)
    barrier(world)
    torch.cuda.synchronize(dev)
    w1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(w0, w1)

    elapsed = ev[0][0].elapsed_time(ev[-1][1]) * 1e-3
    kernel_times = [s.elapsed_time(e) * 1e-3 for s, e in ev]
    kernel_avg = sum(kernel_times) / len(kernel_times)
    elapsed_max = max_over_ranks(elapsed, world)
    updates_per_step = T * HV
    value = world * updates_per_step * args.steps / elapsed_max

    # End to end through the C ABI with host buffers, every step: the step's
    # inputs copied from pinned host memory and its output read back into
    # pinned host memory.  The copies run on a second stream into
    # double-buffered device inputs, overlapping the previous step's kernel;
    # the host waits for each step's output one step behind (a serving loop).
    keys = ("q", "k", "v", "raw_gate", "beta_logits", "cu_seqlens", "state_indices")
    host = {k: inp[k].pin_memory() for k in keys}
    dev_in = [{k: torch.empty_like(host[k], device=dev) for k in keys} for _ in range(2)]
    dev_out = [torch.empty(T, HV, V, device=dev) for _ in range(2)]
    host_out = [torch.empty(T, HV, V, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    copy_stream = torch.cuda.Stream(dev)
    out_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(computed[b])  # step i - 2's kernel is done with this buffer
            for k in keys:
                dev_in[b][k].copy_(host[k], non_blocking=True)
            copied[b].record(copy_stream)

    def run_e2e(n):
        copy_in(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                copy_in(i + 1)
            stream.wait_event(copied[b])
            if i >= 2:
                stream.wait_event(done[b])  # step i - 2's output has left this buffer
            kda_decode(dev_out[b], dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"],
                       dev_in[b]["raw_gate"], dev_in[b]["beta_logits"], d["a_log"], d["dt_bias"],
                       dev_in[b]["cu_seqlens"], d["state_pool"], dev_in[b]["state_indices"],
                       gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"],
                       dev_status=status, stream=stream)
            computed[b].record(stream)
            with torch.cuda.stream(out_stream):  # read back while the next step computes
                out_stream.wait_event(computed[b])
                host_out[b].copy_(dev_out[b], non_blocking=True)
                done[b].record(out_stream)
            if i >= 1:
                done[(i - 1) % 2].synchronize()  # the host has step i - 1's output
        done[(n - 1) % 2].synchronize()

    e2e_steps = max(3, min(args.steps, 200))
    run_e2e(3)
    barrier(world)
    torch.cuda.synchronize(dev)
    w_e0 = time.perf_counter()
    run_e2e(e2e_steps)
    e2e_elapsed = max_over_ranks(time.perf_counter() - w_e0, world)
    e2e_value = world * updates_per_step * e2e_steps / e2e_elapsed

    block = run_block(steps=max(5, min(args.steps, 50)), warmup=3) if rank == 0 else None
    block_n4 = run_block(steps=max(5, min(args.steps, 50)), warmup=3, n=4) if rank == 0 else None
    variant = run_decode_variant(inp, d, steps=max(5, min(args.steps, 200))) if rank == 0 else None
    varlen = run_decode_varlen(steps=max(5, min(args.steps, 200))) if rank == 0 else None
    prefill = run_prefill(steps=3, warmup=1) if rank == 0 else None

    if rank != 0:
        return
    nbytes = decode_bytes(B, T, H, HV, K, V)
    peak, peak_src = measured_peaks()
    achieved = nbytes / kernel_avg / 1e9
    traffic = None
    if NCU_TRAFFIC["sources_sha256"] == kernel_sources_sha():
        traffic = NCU_TRAFFIC["bytes_per_launch"]
    cpu = cpu_baseline(inp) if world == 1 else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * elapsed_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64; bf16 q/k/v, fp32 gates/state)",
        "config": config_dict(cfg),
        "output_tokens_per_s": world * T * args.steps / elapsed_max,
        "hbm_gbs": nbytes / (elapsed_max / args.steps) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6800 GB/s", "algorithmic_bytes_per_launch": nbytes,
                     "kernel": "kda_decode_kernel", "kernel_avg_us": kernel_avg * 1e6},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "note": "every step: pinned host q/k/v/raw_gate/beta_logits/cu_seqlens/"
                        "state_indices copied in (own stream, double-buffered, overlapping "
                        "the previous step's kernel) and the output copied back to pinned host "
                        "memory (own stream, overlapping the next step's kernel), the host "
                        "waiting for each step's output one step behind; "
                        "wall-clock time; state pool and model parameters resident on the device"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "block_tkg": block,
        "block_tkg_n4": block_n4,
        "decode_v_first_bf16": variant,
        "decode_varlen": varlen,
        "prefill": prefill,
    }
    print(json.dumps(line), flush=True)


def run_profile_case(args, which: str):
    """A reduced case for ncu captures: the decode kernel on B = 32 requests x
    1 token, H = 48, HV = 96 (a 64-slot, 400 MB pool; 200 MB of state traffic
    per launch, above the L2 size), with K-first tiles ("decode") or V-first
    tiles ("decode_vfirst", fp32 output), the full varlen workload (64
    requests of 1..8 tokens, the multi-token kernel: "varlen"), or the block at
    its full size with n = 1 or 4 tokens per request ("block", "block_n4";
    "*_eager": eager calls only, no CUDA graph).
    Prints the median kernel time only."""
    from kda_decode_recurrence_gb300 import STATE_V_FIRST, kda_decode_ex
    dev = torch.device("cuda", 0)
    if which in ("block", "block_n4"):
        n = 4 if which == "block_n4" else 1
        print(json.dumps({"profile": which, **run_block(args.steps, args.warmup, n)}))
        return
    if which in ("block_eager", "block_n4_eager"):
        n = 4 if which == "block_n4_eager" else 1
        print(json.dumps({"profile": which, **run_block_eager(args.steps, args.warmup, n)}))
        return
    if which == "prefill":
        print(json.dumps({"profile": "prefill", **run_prefill(args.steps, args.warmup)}))
        return
    if which == "varlen":
        inp = decode_inputs(DECODE_CONFIGS["varlen"])
    else:
        inp = decode_inputs(DECODE_CONFIGS[WORKLOAD], B=32, max_slots=64)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty(inp["T"], inp["HV"], inp["V"], device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    times = []
    for i in range(args.warmup + args.steps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        kda_decode_ex(out, d["q"], d["k"], d["v"], d["raw_gate"], d["beta_logits"], d["a_log"],
                      d["dt_bias"], d["cu_seqlens"], d["state_pool"], d["state_indices"],
                      gate_mode=inp["gate_mode"], lower_bound=inp["lower_bound"],
                      state_layout=STATE_V_FIRST if which == "decode_vfirst" else 0,
                      dev_status=status)
        e.record()
        e.synchronize()
        if i >= args.warmup:
            times.append(s.elapsed_time(e) * 1e-3)
    t = statistics.median(times)
    nbytes = decode_bytes(inp["B"], inp["T"], inp["H"], inp["HV"], inp["K"], inp["V"])
    print(json.dumps({"profile": which, "B": inp["B"], "us": t * 1e6,
                      "algorithmic_bytes": nbytes, "gbs": nbytes / t / 1e9}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", choices=["decode", "decode_vfirst", "varlen", "block", "block_n4",
                                          "block_eager", "block_n4_eager", "prefill"],
                    default=None,
                    help="run a reduced case of one kernel for ncu (no JSON bench line)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="kda", choices=["kda", "reference"])
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.steps = max(args.steps, 1)
    if args.profile:
        run_profile_case(args, args.profile)
        return
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
