"""The float64 oracle on several host cores: contiguous request ranges, one
per worker process.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the benchmark's CPU
baseline and reference legs use it to time the oracle on all host cores.  The
oracle itself stays single-threaded and unchanged; requests (and, in the
block, rows of a request) are independent, so splitting them over processes
changes no result.

Workers are started once with the "spawn" method (never forked from a
process that may hold a CUDA context) and reused.  Inputs reach them as .npy
files in a temporary directory, memory-mapped on their side; for each pass a
worker widens its range to float64, waits on a barrier with the others, then
runs and times its oracle call, so the wall time measured (first start to
last end) covers the parallel oracle work alone.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import queue
import shutil
import tempfile
import time

import numpy as np

DECODE_TOKENS = ("q", "k", "v", "raw_gate", "beta_logits")
BLOCK_WEIGHTS = ("gamma_in", "W_in", "W_fb", "W_gb", "conv_w", "A_log", "dt_bias", "gamma_o",
                 "W_o")


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _load(dirpath, names):
    return {k: np.load(os.path.join(dirpath, k + ".npy"), mmap_mode="r") for k in names}


def _decode_range(a, b0, b1, gate_mode, lower_bound):
    """The arguments of one oracle call over requests b0..b1-1 (float64)."""
    cu = np.asarray(a["cu"])
    r0, r1 = int(cu[b0]), int(cu[b1])
    tok = {k: np.asarray(a[k][r0:r1], dtype=np.float64) for k in DECODE_TOKENS}
    return dict(q=tok["q"], k=tok["k"], v=tok["v"], raw_gate=tok["raw_gate"],
                beta_logits=tok["beta_logits"], a_log=np.asarray(a["a_log"], np.float64),
                dt_bias=np.asarray(a["dt_bias"], np.float64),
                cu_seqlens=(cu[b0:b1 + 1] - cu[b0]).astype(np.int32),
                state_pool=np.asarray(a["pool"][b0:b1], dtype=np.float64),
                state_indices=np.arange(b1 - b0, dtype=np.int32), gate_mode=gate_mode,
                lower_bound=lower_bound)


def _block_range(a, b0, b1, scalars):
    w = [np.asarray(a[k], dtype=np.float64) for k in BLOCK_WEIGHTS]
    return ([np.asarray(a["hidden"][b0:b1], np.float64)] + w +
            [np.asarray(a["S"][b0:b1], np.float64),
             np.asarray(a["conv_state"][b0:b1], np.float64)] + list(scalars))


def _prepare(kind, dirpath, b0, b1, extra, cache):
    if kind == "decode":
        a = cache.setdefault(dirpath, _load(dirpath, DECODE_TOKENS + ("a_log", "dt_bias", "cu", "pool")))
        return _decode_range(a, b0, b1, *extra)
    a = cache.setdefault(dirpath, _load(dirpath, BLOCK_WEIGHTS + ("hidden", "S", "conv_state")))
    return _block_range(a, b0, b1, extra)


def _call(kind, args):
    import oracle
    if kind == "decode":
        oracle.kda_decode(**args)
    else:
        oracle.kda_block_tkg(*args)


def _loop(tasks, barrier, results, slot):
    """Worker: take (kind, dirpath, b0, b1, extra) tasks until None; for each,
    prepare its range, meet the other workers at the barrier, then run and
    time the oracle on it."""
    cache = {}
    while True:
        task = tasks.get()
        if task is None:
            return
        kind, dirpath, b0, b1, extra = task
        try:
            args = _prepare(kind, dirpath, b0, b1, extra, cache) if b1 > b0 else None
        except Exception as e:  # let the others through the barrier, then report
            barrier.abort()
            results.put((slot, None, repr(e)))
            continue
        try:
            barrier.wait(timeout=600)
        except Exception as e:
            results.put((slot, None, repr(e)))
            continue
        t0 = time.time()
        if args is not None:
            _call(kind, args)
        results.put((slot, t0, time.time()))


class OracleWorkers:
    """`n` spawned worker processes that run the oracle on request ranges in
    parallel.  Use as a context manager; stage() writes a workload's arrays
    once, run() times one pass of the oracle over its first n_requests."""

    def __init__(self, n: int):
        self.n = max(1, int(n))
        ctx = mp.get_context("spawn")
        self.barrier = ctx.Barrier(self.n)
        self.results = ctx.Queue()
        self.tasks = [ctx.Queue() for _ in range(self.n)]
        self.procs = [ctx.Process(target=_loop, args=(self.tasks[i], self.barrier, self.results, i),
                                  daemon=True) for i in range(self.n)]
        for p in self.procs:
            p.start()
        self.dirs = []

    def stage(self, arrays: dict) -> str:
        d = tempfile.mkdtemp(prefix="kda_oracle_")
        for k, v in arrays.items():
            np.save(os.path.join(d, k + ".npy"), np.ascontiguousarray(v))
        self.dirs.append(d)
        return d

    def run(self, kind: str, dirpath: str, n_requests: int, extra) -> float:
        edges = [round(i * n_requests / self.n) for i in range(self.n + 1)]
        for i in range(self.n):
            self.tasks[i].put((kind, dirpath, edges[i], edges[i + 1], tuple(extra)))
        got = []
        deadline = time.time() + 1800
        while len(got) < self.n:
            try:
                got.append(self.results.get(timeout=1.0))
            except queue.Empty:
                dead = [p.exitcode for p in self.procs if not p.is_alive()]
                if dead or time.time() > deadline:
                    raise RuntimeError(f"oracle workers stopped (exit codes {dead})")
        bad = [g for g in got if g[1] is None]
        if bad:
            self.barrier.reset()
            raise RuntimeError(f"oracle worker failed: {bad[0][2]}")
        return max(t1 for _, _, t1 in got) - min(t0 for _, t0, _ in got)

    def close(self):
        for q in self.tasks:
            q.put(None)
        for p in self.procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
        for d in self.dirs:
            shutil.rmtree(d, ignore_errors=True)
        self.dirs = []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def decode_arrays(tokens: dict, a_log, dt_bias, cu_seqlens, pool_rows) -> dict:
    """A decode workload as the workers read it.  tokens: q, k, v, raw_gate,
    beta_logits (packed by token, any float dtype); pool_rows: the requests'
    state tiles in request order [B, HV, K, V]."""
    arrays = {k: tokens[k] for k in DECODE_TOKENS}
    arrays.update(a_log=a_log, dt_bias=dt_bias, cu=np.asarray(cu_seqlens, np.int64),
                  pool=pool_rows)
    return arrays


def block_arrays(params: dict, hidden, S, conv_state) -> dict:
    arrays = {k: params[k] for k in BLOCK_WEIGHTS}
    arrays.update(hidden=hidden, S=S, conv_state=conv_state)
    return arrays


def time_single(kind: str, arrays: dict, n_requests: int, extra) -> float:
    """The same pass in this process, one thread (inputs widened first)."""
    a = {k: np.asarray(v) for k, v in arrays.items()}
    args = (_decode_range(a, 0, n_requests, *extra) if kind == "decode"
            else _block_range(a, 0, n_requests, extra))
    t0 = time.perf_counter()
    _call(kind, args)
    return time.perf_counter() - t0
