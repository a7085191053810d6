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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="decode_gqa")
    ap.add_argument("--seconds", type=float, default=15.0)
    a = ap.parse_args()
    import kvq_workloads as W
    inp = W.NAMED[a.workload]()
    if a.workload.startswith("prefill"):
        r = time_prefill(inp, a.seconds)
    else:
        r = time_decode(inp, a.seconds)
    r["cores"] = int(os.environ.get("OMP_NUM_THREADS", "0") or 0) or os.cpu_count()
    r["kind"] = "oracle"
    print(json.dumps(r))


if __name__ == "__main__":
    main()
