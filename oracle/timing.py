"""Times the CPU oracle, as it stands, on a bounded sample of a workload.

TEST/BENCHMARK INFRASTRUCTURE: run only by the benchmark's CPU-baseline leg
and reference arm (as a subprocess, so thread counts can be pinned through
the environment).  Prints one JSON object.

Units match the benchmark's metric: algorithmic cache bytes (codes + scale
and zero words of K and V) that the oracle consumed per second, for decode;
algorithmic FLOP per second for prefill.  The oracle's work per unit is the
whole method: quantise the bf16 K/V rows, dequantise, attend.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import kvq_oracle as O  # noqa: E402


def time_decode(inp, seconds: float):
    """Run the oracle over (sequence, KV head) segments in order until `seconds` pass."""
    B, Hq, Hkv, D = inp.B, inp.Hq, inp.Hkv, inp.D
    rep = Hq // Hkv
    done_bytes = 0
    segs = 0
    t0 = time.perf_counter()
    for b in range(B):
        L = int(inp.seq_lens[b])
        for kv in range(Hkv):
            bits = int(inp.head_bits[kv])
            kc, ks, kz = O.quantize_groups(inp.k[b, kv, :L], bits)
            vc, vs, vz = O.quantize_groups(inp.v[b, kv, :L], bits)
            kd, vd = O.dequantize(kc, ks, kz), O.dequantize(vc, vs, vz)
            q = O.bf16_to_f32(inp.q[b, kv * rep:(kv + 1) * rep]).astype(np.float64)
            O.attention(q, kd, vd, inp.softmax_scale)
            done_bytes += 2 * L * (D * bits // 8 + 4 * (D // 32))
            segs += 1
            if time.perf_counter() - t0 > seconds:
                break
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": done_bytes / dt / 1e9, "unit": "GB/s", "seconds": dt,
            "sample": f"{segs} of {B * Hkv} (sequence, KV head) segments of {inp.name}: "
                      f"oracle quantise + dequantise + attention of all {rep} query heads"}


def time_prefill(inp, seconds: float, rows_per_head: int = 64):
    """Oracle prefill on evenly spaced query rows of successive heads until `seconds` pass."""
    B, Hq, Hkv, S, D = inp.B, inp.Hq, inp.Hkv, inp.S, inp.D
    rep = Hq // Hkv
    flops = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    deq = {}
    for h in range(Hq):
        kv = h // rep
        if kv not in deq:
            kc, ks, kz = O.quantize_groups(inp.k[0, kv], 8)
            vc, vs, vz = O.quantize_groups(inp.v[0, kv], 8)
            deq = {kv: (O.dequantize(kc, ks, kz)[None, None], O.dequantize(vc, vs, vz)[None, None])}
        kd, vd = deq[kv]
        rows = np.linspace(0, S - 1, rows_per_head).astype(np.int64)
        for r in rows:
            O.prefill_rows(inp.q, kd, vd, 0, h, np.array([r]), inp.tile_mask, inp.softmax_scale)
            allowed = O.prefill_allowed(np.array([r]), int(r) + 1, inp.tile_mask)
            flops += 4.0 * D * float(allowed.sum())
            rows_done += 1
            if time.perf_counter() - t0 > seconds:
                break
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "seconds": dt,
            "sample": f"{rows_done} query rows (evenly spaced, successive heads) of {inp.name}, "
                      f"with the oracle's K/V quantise + dequantise of each KV head"}


# ----------------------------------------------------------------------------
# several host cores: one worker process per core, each taking every procs-th
# (sequence, KV head) segment of the same workload
# ----------------------------------------------------------------------------

_WORKER_INP = None


def _worker_init(workload: str):
    global _WORKER_INP
    import kvq_workloads as W
    _WORKER_INP = W.NAMED[workload]()


def _segment_bytes(inp, b: int, kv: int) -> int:
    return 2 * int(inp.seq_lens[b]) * (inp.D * int(inp.head_bits[kv]) // 8 + 4 * (inp.D // 32))


def _worker_run(args):
    """Oracle quantise + dequantise + attention of segments r, r + procs, ...
    (cyclically) until `seconds` pass; returns (bytes, seconds, segments)."""
    r, procs, seconds = args
    inp = _WORKER_INP
    rep = inp.Hq // inp.Hkv
    n_seg = inp.B * inp.Hkv
    done, segs, i = 0, 0, r
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        b, kv = divmod(i % n_seg, inp.Hkv)
        L = int(inp.seq_lens[b])
        bits = int(inp.head_bits[kv])
        kc, ks, kz = O.quantize_groups(inp.k[b, kv, :L], bits)
        vc, vs, vz = O.quantize_groups(inp.v[b, kv, :L], bits)
        q = O.bf16_to_f32(inp.q[b, kv * rep:(kv + 1) * rep]).astype(np.float64)
        if L > 0:
            O.attention(q, O.dequantize(kc, ks, kz), O.dequantize(vc, vs, vz), inp.softmax_scale)
        done += _segment_bytes(inp, b, kv)
        segs += 1
        i += procs
    return done, time.perf_counter() - t0, segs


class ParallelDecodeTimer:
    """A pool of `procs` spawned worker processes (BLAS pinned to one thread
    each), each holding the workload once; ``step(seconds)`` runs them all for
    about that long and returns the aggregate oracle GB/s.  Spawned, not
    forked, so it is safe to start from a process that has touched a GPU."""

    def __init__(self, workload: str, procs: int):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.procs = procs
        self.workload = workload
        self.pool = mp.get_context("spawn").Pool(procs, initializer=_worker_init, initargs=(workload,))

    def step(self, seconds: float) -> dict:
        res = self.pool.map(_worker_run, [(r, self.procs, seconds) for r in range(self.procs)])
        total = sum(x[0] for x in res)
        dt = max(x[1] for x in res)
        segs = sum(x[2] for x in res)
        return {"value": total / dt / 1e9, "unit": "GB/s", "seconds": dt, "cores": self.procs,
                "sample": f"{segs} (sequence, KV head) segments of {self.workload} over {self.procs} worker "
                          f"processes (one per host core, BLAS one thread each): oracle quantise + dequantise + "
                          f"attention of every query head of a segment"}

    def close(self):
        self.pool.close()
        self.pool.join()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="decode_gqa")
    ap.add_argument("--seconds", type=float, default=15.0)
    ap.add_argument("--procs", type=int, default=1,
                    help="decode only: worker processes (0 = every host core)")
    a = ap.parse_args()
    import kvq_workloads as W
    # one process: as many cores as its BLAS may use (the benchmark pins it to 1)
    one = int(os.environ.get("OMP_NUM_THREADS", "0") or 0) or (os.cpu_count() or 1)
    if a.workload.startswith("prefill"):
        r = time_prefill(W.NAMED[a.workload](), a.seconds)
        r["cores"] = one
    elif a.procs != 1:
        t = ParallelDecodeTimer(a.workload, a.procs if a.procs > 0 else (os.cpu_count() or 1))
        try:
            r = t.step(a.seconds)
        finally:
            t.close()
    else:
        r = time_decode(W.NAMED[a.workload](), a.seconds)
        r["cores"] = one
    r["kind"] = "oracle"
    print(json.dumps(r))


if __name__ == "__main__":
    main()
