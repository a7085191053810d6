"""Benchmark: quantised-KV decode attention HBM GB/s on one GB300 (per rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference]
                    [--workload decode_gqa] [--no-cpu-baseline] [--no-prefill]

A step is one decode-attention call (split-K pass with its log-sum-exp merge)
of the whole batch over its quantised cache, resident in HBM; the cache is
quantised once, untimed, by kvq_quantize.  Several copies of the cache (more
than 3x L2 together) are visited in turn, so no step finds its bytes in L2,
and the timed steps run back to back between one pair of CUDA events.  ``value``
is algorithmic cache bytes (codes plus scale/zero words of K and V) per
second over all ranks.  Under torchrun each rank runs its own batch
(independent sequences: weak scaling, no collective on the data path).

Also reported: ``e2e`` (the same metric through the C ABI with the step's
new inputs copied from pinned host memory and the output read back every
step), ``roofline`` for the split kernel, the CPU oracle timed on a bounded
sample (``cpu_baseline``), clocks sampled during the timed region, and the
causal and non-causal prefill workloads' TFLOP/s when the prefill kernel is available.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# the one metric string both arms print, so their lines can be paired
METRIC = "quant-KV decode attn HBM GB/s (% of peak); prefill attn TFLOP/s (% of peak)"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    found = {}
    if os.path.exists(path):
        try:
            data = json.load(open(path))

            def walk(d):
                if isinstance(d, dict):
                    for k, v in d.items():
                        if isinstance(v, (int, float)) and k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                            found.setdefault(k, float(v))
                        else:
                            walk(v)
                elif isinstance(d, list):
                    for v in d:
                        walk(v)
            walk(data)
        except Exception:
            found = {}
    hbm = found.get("hbm_gbs")
    bf = found.get("bf16_tflops")
    bfs = found.get("bf16_tflops_sustained")
    return {
        "hbm_gbs": hbm or FALLBACK_HBM_GBS, "hbm_src": "of measured" if hbm else "of fallback",
        "bf16_tflops": bf or FALLBACK_BF16_TFLOPS, "bf16_src": "of measured" if bf else "of fallback",
        "bf16_tflops_sustained": bfs or bf or 1700.0,
    }


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _traffic_from_profile(kernel_src: str, workload: str):
    """DRAM bytes per launch recorded by the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if "=" in line and not line.lstrip().startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    src = open(os.path.join(ROOT, "attention_group_quantized_gb300", "csrc", kernel_src), "rb").read()
    if kv.get("source_sha256") != hashlib.sha256(src).hexdigest():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _oracle_subprocess(workload: str, seconds: float, procs: int = 1):
    """The CPU oracle timed on a bounded sample, in a child process (BLAS one
    thread per process; procs = 0 runs one worker process per host core)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "oracle.timing", "--workload", workload, "--seconds", str(seconds),
                        "--procs", str(procs)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1:] or ["failed"]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def _cpu_entry(r: dict) -> dict:
    if "error" in r:
        return r
    return {"value": r["value"], "unit": r["unit"], "cores": r["cores"], "kind": "oracle", "sample": r["sample"]}


def _p95(xs):
    """95th percentile of a few samples (nearest rank)."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, int(0.95 * len(ys) + 0.5) - 1)] if ys else float("nan")


def max_over_ranks(torch, dist, value: float, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if not dist:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_step: int, world: int, steps: int, t_max: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_step per step (weak scaling)."""
    return bytes_per_step * world * steps / t_max / 1e9


def decode_bytes(inp) -> int:
    D = inp.D
    tot = 0
    for b in range(inp.B):
        for h in range(inp.Hkv):
            tot += 2 * int(inp.seq_lens[b]) * (D * int(inp.head_bits[h]) // 8 + 4 * (D // 32))
    return tot


def run_reference(args, rank):
    """Reference arm: the CPU oracle, as it stands, on the host cores (rank 0
    only).  A step is a bounded sample of the decode workload, run by one
    worker process per host core; the prefill workload's oracle is timed once
    beside it on one core."""
    if rank != 0:
        return
    import kvq_workloads as W
    from oracle import timing as OT
    name = W.NAMED[args.workload]().name
    per_step = getattr(args, "step_seconds", None) or max(2.0, 60.0 / max(1, args.steps + args.warmup))
    procs = os.cpu_count() or 1
    try:
        timer = OT.ParallelDecodeTimer(args.workload, procs)
    except Exception as e:   # no process pool on this host
        print(json.dumps({"impl": "reference", "unavailable": f"oracle worker pool failed: {e}"}))
        return
    vals = []
    last = None
    try:
        for i in range(args.warmup + args.steps):
            r = timer.step(per_step)
            if i >= args.warmup:
                vals.append(r["value"])
            last = r
    finally:
        timer.close()
    v = statistics.mean(vals)
    pre = _oracle_subprocess("prefill_causal", 10.0)
    prefill = None
    if "error" not in pre:
        prefill = {"workload": W.NAMED["prefill_causal"]().name, "value": pre["value"], "unit": pre["unit"],
                   "cpu_baseline": _cpu_entry(pre)}
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded, kvq_workloads)",
            "config": {"workload": name},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"]},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "prefill": prefill}
    print(json.dumps(line))


def time_decode(torch, kvq, inp, dev, l2, steps, warmup, dist=None, keep=False, busy_s=0.0, sampler=None,
                use_graph=True, paged=False, policy=None):
    """Back-to-back decode steps over cache copies larger than 3x L2 together.

    With paged=True each copy is a pair of page pools addressed through a
    shuffled block table (kvq_decode_attention_paged).  Returns the total
    device time of `steps` steps (max over ranks) and the algorithmic bytes
    per step; with keep=True also the device buffers.
    """
    import numpy as np
    B, Hq, Hkv, D, Tcap = inp.B, inp.Hq, inp.Hkv, inp.D, inp.Tcap
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    nbytes = decode_bytes(inp)
    n_copies = max(2, -(-3 * l2 // max(nbytes, 1)))
    kd, vd = todev(inp.k), todev(inp.v)
    caches = []
    tables = []
    for c in range(n_copies):
        if paged:
            max_pages = Tcap // 64
            n_pages = B * max_pages
            perm = np.random.default_rng(100 + c).permutation(n_pages).astype(np.int32)
            bt = torch.from_numpy(perm.reshape(B, max_pages)).to(dev)
            kc = kvq.empty_page_pool(inp.head_bits, n_pages, D, device=dev)
            vc = kvq.empty_page_pool(inp.head_bits, n_pages, D, device=dev)
            kvq.quantize_paged(kd, kc, bt)
            kvq.quantize_paged(vd, vc, bt)
            tables.append(bt)
        else:
            kc = kvq.empty_cache(inp.head_bits, B, Tcap, D, device=dev)
            vc = kvq.empty_cache(inp.head_bits, B, Tcap, D, device=dev)
            kvq.quantize(kd, kc)
            kvq.quantize(vd, vc)
        caches.append((kc, vc))
    del kd, vd
    q = todev(inp.q)
    sl = torch.from_numpy(inp.seq_lens).to(dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = kvq.decode_workspace(B, Hq, Hkv, D, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        kc_i, vc_i = caches[i % n_copies]
        if paged:
            kvq.decode_attention_paged(q, kc_i, vc_i, tables[i % n_copies], sl, inp.softmax_scale, out=out,
                                       workspace=ws, status=status)
        else:
            kvq.decode_attention(q, kc_i, vc_i, sl, inp.softmax_scale, out=out, workspace=ws, status=status,
                                 policy=policy)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    clk = sampler() if sampler else None
    if clk:
        clk.__enter__()
    # sustained load (untimed) right before the timed steps, so clock samples
    # taken around them see the GPU in the same state
    t_busy = time.time()
    while time.time() - t_busy < busy_s:
        for i in range(200):
            step(i)
        torch.cuda.synchronize()
    # the K timed steps as one CUDA graph (launches captured with their
    # programmatic-dependency edges), so host launch jitter stays out of the
    # device time; replayed once untimed first (graph upload)
    graph = None
    if use_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(steps):
                    step(i)
            graph.replay()
            torch.cuda.synchronize()
        except Exception as e:   # capture unsupported here: time the eager loop
            print(f"bench: CUDA graph capture failed ({e}); timing eager launches", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(steps):
            step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if clk:
        clk.__exit__(None, None, None)
    t_total = max_over_ranks(torch, dist, t0.elapsed_time(t1) / 1e3, dev)
    # isolated launches (each synchronised before the next): no overlap with a
    # previous kernel, so the launch ramp and the merge tail are not hidden.
    # iso: events around the call, so the host's enqueue (the GPU idles
    # meanwhile) is included; iso_dev: a spin kernel queued first keeps the
    # GPU busy while the call is enqueued, so the events bracket the device
    # work of the launch alone
    iso, iso_dev = [], []
    for i in range(min(steps, 10)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        iso.append(e0.elapsed_time(e1) * 1e3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200000)   # about 0.1 ms of device spin
        e0.record(stream)
        step(i + 1)
        e1.record(stream)
        torch.cuda.synchronize()
        iso_dev.append(e0.elapsed_time(e1) * 1e3)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    res = {"t_total": t_total, "bytes": nbytes, "n_copies": n_copies, "clk": clk,
           "isolated_us": statistics.median(iso), "isolated_device_us": statistics.median(iso_dev),
           "timing": "one CUDA graph of the K steps, event-timed" if graph is not None else "eager launches, event-timed"}
    if keep:
        res.update(caches=caches, q=q, sl=sl, ws=ws)
    return res


def bench_extra_decodes(torch, kvq, W, peaks, dev, steps, warmup):
    """The other decode workloads, measured the same way (context for the main line)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    for name, paged in (("decode_long_ragged", False), ("decode_mixed", False), ("decode_tiny", False),
                        ("decode_gqa", True)):
        inp = W.NAMED[name]()
        d = time_decode(torch, kvq, inp, dev, l2, steps, warmup, paged=paged)
        avg = d["t_total"] / steps
        gbs = d["bytes"] / avg / 1e9
        key = inp.name + ("_paged_shuffled_block_table" if paged else "")
        res[key] = {"GB/s": round(gbs, 1), "us_per_step": round(avg * 1e6, 2),
                         "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4), "bytes_per_step": d["bytes"]}
        del d
        torch.cuda.empty_cache()
    res["decode_tiny_with_quantize"] = time_tiny_with_quantize(torch, kvq, W, dev, steps, warmup)
    return res


def time_tiny_with_quantize(torch, kvq, W, dev, steps, warmup):
    """decode_tiny as its configuration states it: each step quantises the 512-token K and V into the
    caches and then decodes (three launches), steps back to back in one CUDA graph."""
    import numpy as np
    inp = W.decode_tiny()
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    k, v, q = todev(inp.k), todev(inp.v), todev(inp.q)
    kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D, device=dev)
    vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D, device=dev)
    sl = torch.from_numpy(inp.seq_lens).to(dev)
    out = torch.empty((inp.B, inp.Hq, inp.D), dtype=torch.float32, device=dev)
    ws = kvq.decode_workspace(inp.B, inp.Hq, inp.Hkv, inp.D, dev)

    def step():
        kvq.quantize(k, kc)
        kvq.quantize(v, vc)
        kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, out=out, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            step()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / steps
    kv_bytes = 2 * inp.B * inp.Hkv * inp.Tcap * (inp.D + 4 * inp.D // 32)
    q_bytes = 2 * (2 * inp.B * inp.Hkv * inp.Tcap * inp.D) + kv_bytes
    return {"us_per_step": round(us, 2), "launches_per_step": 3,
            "bytes_per_step": {"quantize": q_bytes, "decode": kv_bytes},
            "note": "latency workload: quantise K and V (bf16 in, codes and scale/zero words out), then decode"}


def bench_quantize(torch, kvq, inp, peaks, steps, warmup, dev):
    """kvq_quantize on the decode workload's K tensor ([B][Hkv][T][D] bf16 -> codes + scale/zero words):
    HBM bytes = bf16 read + codes and words written, two input copies visited in turn (each larger
    than L2), calls back to back between CUDA events."""
    import numpy as np
    B, Hkv, T, D = inp.B, inp.Hkv, inp.Tcap, inp.D
    x0 = torch.from_numpy(np.ascontiguousarray(inp.k).view(np.int16)).view(torch.bfloat16).to(dev)
    xs = [x0, x0.clone()]
    cache = kvq.empty_cache(inp.head_bits, B, T, D, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rd = x0.numel() * 2
    wr = sum(B * T * D * int(b) // 8 for b in inp.head_bits) + B * Hkv * T * (D // 32) * 4
    for i in range(warmup):
        kvq.quantize(xs[i % 2], cache, 0, status)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        kvq.quantize(xs[i % 2], cache, 0, status)
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    t = e0.elapsed_time(e1) / 1e3 / steps
    gbs = (rd + wr) / t / 1e9
    return {"workload": f"quantize {inp.name} K ({B}x{Hkv}x{T}x{D} bf16)", "value": gbs, "unit": "GB/s",
            "us_per_call": t * 1e6, "bytes_per_call": int(rd + wr), "read_bytes": int(rd), "write_bytes": int(wr),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_src": peaks["hbm_src"]}}


def bench_head_bits(torch, kvq, W, peaks, steps, warmup, dev):
    """Per-head bit allocation on the head_bits workload (decode_gqa's K/V shape, weighted): one step =
    kvq_head_error_stats of K and of V (two launches each, the device-side part) back to back between CUDA
    events; K and V are visited in turn, together larger than L2.  HBM bytes = the bf16 rows + the float
    weights read by each call.  The host allocation (a sort of H scores) is timed apart, after the
    statistics are copied back."""
    import numpy as np
    inp = W.head_bits_kv()
    B, H, T, D = inp.k.shape
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    k, v = todev(inp.k), todev(inp.v)
    w = torch.from_numpy(inp.weights).to(dev)
    ws = kvq.head_error_stats_workspace(H, dev)
    ks = torch.empty((H, 2), dtype=torch.float64, device=dev)
    vs = torch.empty((H, 2), dtype=torch.float64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    step = lambda: (kvq.head_error_stats(k, 4, weights=w, workspace=ws, out=ks, status=status),
                    kvq.head_error_stats(v, 4, weights=w, workspace=ws, out=vs, status=status))
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    t = e0.elapsed_time(e1) / 1e3 / steps / 2            # per call (one tensor)
    per_call = k.numel() * 2 + w.numel() * 4
    gbs = per_call / t / 1e9
    t0 = time.perf_counter()
    bits, _ = kvq.allocate_head_bits(ks, vs, len(inp.outlier_heads))
    alloc_us = (time.perf_counter() - t0) * 1e6
    return {"workload": inp.name, "value": gbs, "unit": "GB/s", "us_per_call": t * 1e6,
            "bytes_per_call": int(per_call), "host_allocation_us": alloc_us,
            "chosen_8bit_heads": [int(h) for h in np.flatnonzero(bits == 8)],
            "outlier_heads": [int(h) for h in inp.outlier_heads],
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_src": peaks["hbm_src"]}}


def bench_phase_policy(torch, kvq, W, peaks, steps, warmup, dev, decode_policy):
    """Phase-specific settings (prefill and decode tuned apart): the causal
    prefill workload with a sparser tile mask -- 35 % of each row's candidate
    key tiles skipped, built on the device by kvq_build_tile_mask -- and the
    decode workload with a wider prefetch policy, each beside the defaults."""
    import numpy as np
    res = {}
    inp = W.prefill_causal()
    B, Hq, S, D = inp.B, inp.Hq, inp.S, inp.D
    n_t = S // 128
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v = todev(inp.q), todev(inp.k), todev(inp.v)
    kc = kvq.empty_cache(inp.head_bits, B, S, D, device=dev)
    vc = kvq.empty_cache(inp.head_bits, B, S, D, device=dev)
    out = torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device=dev)
    for num, den, label in ((1, 4, "skip25_builder"), (7, 20, "skip35_builder")):
        mask = kvq.build_tile_mask(n_t, num, den, 4, device=dev)
        m = mask.cpu().numpy()
        kept = int(np.tril(m, -1).sum())
        flops = 4.0 * D * Hq * B * (kept * 128 * 128 + n_t * 128 * 129 / 2)
        run = lambda: kvq.prefill_attention(q, k, v, kc, vc, inp.softmax_scale, mask, out=out, out_dtype=kvq.OUT_BF16)
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            run()
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / steps
        res[label] = {"skipped_share_of_row_candidates": f"{num}/{den}", "kept_below_diagonal_tiles": kept,
                      "ms_per_step": t * 1e3, "algorithmic_flop": flops, "TFLOP/s": flops / t / 1e12,
                      "frac_of_bf16_peak": flops / t / 1e12 / peaks["bf16_tflops"]}
    res["prefill_speedup_35_over_25"] = res["skip25_builder"]["ms_per_step"] / res["skip35_builder"]["ms_per_step"]
    del q, k, v, kc, vc, out
    torch.cuda.empty_cache()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    dinp = W.decode_gqa()
    variants = (("decode_ring2", {"decode_ring_tiles": 2}), ("decode_default", {}),
                ("decode_policy", dict(decode_policy)))
    for label, fields in variants:
        d = time_decode(torch, kvq, dinp, dev, l2, steps, warmup, policy=kvq.policy(**fields) if fields else None)
        avg = d["t_total"] / steps
        res[label] = {"policy": fields or "defaults (ring 4, L2 warm-up 5)",
                      "us_per_step": avg * 1e6, "isolated_launch_us": d["isolated_us"],
                      "isolated_device_us": d["isolated_device_us"],
                      "GB/s": d["bytes"] / avg / 1e9, "frac_of_hbm_peak": d["bytes"] / avg / 1e9 / peaks["hbm_gbs"]}
        del d
    res["decode_speedup_policy_over_default"] = res["decode_default"]["us_per_step"] / res["decode_policy"]["us_per_step"]
    return res


def bench_prefill_varlen(torch, kvq, W, peaks, steps, warmup, dev):
    """Causal prefill of 4 sequences of different lengths padded to one S (kvq_prefill_attention_varlen):
    TFLOP/s of the work the lengths ask for, 4 * D * Hq * sum_b L_b (L_b + 1) / 2."""
    import numpy as np
    inp, lens = W.prefill_varlen()
    B, Hq, Hkv, S, D = inp.B, inp.Hq, inp.Hkv, inp.S, inp.D
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v = todev(inp.q), todev(inp.k), todev(inp.v)
    sl = torch.from_numpy(lens).to(dev)
    kc = kvq.empty_cache(inp.head_bits, B, S, D, device=dev)
    vc = kvq.empty_cache(inp.head_bits, B, S, D, device=dev)
    out = torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device=dev)
    run = lambda: kvq.prefill_attention(q, k, v, kc, vc, inp.softmax_scale, None, out=out, out_dtype=kvq.OUT_BF16,
                                        seq_lens=sl)
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / steps
    flops = 4.0 * D * Hq * float(sum(int(L) * (int(L) + 1) / 2 for L in lens))
    tf = flops / t / 1e12
    return {"workload": inp.name, "lengths": [int(L) for L in lens], "value": tf, "unit": "TFLOP/s",
            "ms_per_step": t * 1e3, "algorithmic_flop": flops,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "peak_src": peaks["bf16_src"],
                         "note": "time includes the two quantise launches; causal work only (no padding)"}}


def bench_prefill(torch, kvq, W, peaks, steps, warmup, dev, causal=True):
    """Prefill workload (quantise K/V + attention): TFLOP/s.  Causal: the
    tile-masked causal workload; non-causal: the same shapes, every key visible,
    no mask."""
    import numpy as np
    inp = W.prefill_causal() if causal else W.prefill_noncausal()
    B, Hq, Hkv, S, D = inp.B, inp.Hq, inp.Hkv, inp.S, inp.D
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v = todev(inp.q), todev(inp.k), todev(inp.v)
    mask = torch.from_numpy(inp.tile_mask).to(dev) if inp.tile_mask is not None else None
    run = lambda: kvq.prefill_attention(q, k, v, kc, vc, inp.softmax_scale, mask, out=out, out_dtype=kvq.OUT_BF16,
                                        causal=causal)
    kc = kvq.empty_cache(inp.head_bits, B, S, D, device=dev)
    vc = kvq.empty_cache(inp.head_bits, B, S, D, device=dev)
    out = torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device=dev)
    try:
        run()
    except kvq.KvqError as e:
        return {"unavailable": str(e)}
    n_t = S // 128
    if causal:
        kept = int(np.tril(inp.tile_mask, -1).sum())
        flops = 4.0 * D * Hq * B * (kept * 128 * 128 + n_t * 128 * 129 / 2)
    else:
        flops = 4.0 * D * Hq * B * S * S
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    t = statistics.mean(times)
    tf = flops / t / 1e12
    res = {"workload": inp.name, "value": tf, "unit": "TFLOP/s", "ms_per_step": t * 1e3,
           "ms_median": statistics.median(times) * 1e3, "ms_p95": _p95(times) * 1e3,
           "algorithmic_flop": flops,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": tf / peaks["bf16_tflops"], "peak_src": peaks["bf16_src"],
                        "note": "time includes the two quantise launches of the same call"}}
    if not causal:
        return res
    # the device-side tile-mask builder for this prefill's grid (25 % of the candidate tiles per row)
    for _ in range(3):
        kvq.build_tile_mask(n_t, 1, 4, 4, device=dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        kvq.build_tile_mask(n_t, 1, 4, 4, device=dev)
    e1.record()
    torch.cuda.synchronize()
    mask_us = e0.elapsed_time(e1) * 1e3 / 10
    res["tile_mask_build_us"] = {"nT": n_t, "skip": "1/4 per row", "us": mask_us}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default="decode_gqa")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the other decode workloads")
    ap.add_argument("--busy-seconds", type=float, default=1.0,
                    help="untimed sustained decode steps before the timed ones, under the clock sampler")
    ap.add_argument("--only-prefill", action="store_true",
                    help="run only the prefill workloads (causal, non-causal) and print their JSON object")
    ap.add_argument("--only-head-bits", action="store_true",
                    help="run only the per-head bit allocation workload and print its JSON object")
    ap.add_argument("--only-phase-policy", action="store_true",
                    help="run only the phase-policy legs (sparser prefill mask, wider decode prefetch)")
    ap.add_argument("--decode-policy", default="ring=4,warm=10",
                    help="decode policy timed beside the defaults in the phase-policy leg: ring tiles, L2 warm-up tiles")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import numpy as np
    import torch

    import kvq_workloads as W
    from attention_group_quantized_gb300 import kvq

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    kvq.lib()   # fail loudly if the library is missing
    peaks = _peaks()
    if args.only_head_bits:
        if rank == 0:
            print(json.dumps(bench_head_bits(torch, kvq, W, peaks, args.steps, args.warmup, dev)))
        if dist:
            dist.destroy_process_group()
        return
    pol_fields = dict(kv.split("=") for kv in args.decode_policy.split(","))
    decode_policy = {"decode_ring_tiles": int(pol_fields.get("ring", 4)),
                     "decode_l2_warm_tiles": int(pol_fields.get("warm", 5))}
    if args.only_phase_policy:
        if rank == 0:
            print(json.dumps(bench_phase_policy(torch, kvq, W, peaks, args.steps, args.warmup, dev, decode_policy)))
        if dist:
            dist.destroy_process_group()
        return
    if args.only_prefill:
        if rank == 0:
            res = bench_prefill(torch, kvq, W, peaks, args.steps, args.warmup, dev)
            res["non_causal"] = bench_prefill(torch, kvq, W, peaks, args.steps, args.warmup, dev, causal=False)
            res["varlen"] = bench_prefill_varlen(torch, kvq, W, peaks, args.steps, args.warmup, dev)
            print(json.dumps(res))
        if dist:
            dist.destroy_process_group()
        return

    inp = W.NAMED[args.workload]()
    B, Hq, Hkv, D, Tcap = inp.B, inp.Hq, inp.Hkv, inp.D, inp.Tcap
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    d = time_decode(torch, kvq, inp, dev, l2, args.steps, args.warmup, dist, keep=True, busy_s=args.busy_seconds,
                    sampler=lambda: ClockSampler(local))
    clk = d["clk"]
    timing = d["timing"]
    isolated_us = d["isolated_us"]
    isolated_dev_us = d["isolated_device_us"]
    caches, n_copies, q, sl, ws = d["caches"], d["n_copies"], d["q"], d["sl"], d["ws"]
    bytes_per_step = d["bytes"]
    t_total = d["t_total"]
    value = job_gbs(bytes_per_step, world, args.steps, t_total)
    avg = t_total / args.steps
    achieved = bytes_per_step / avg / 1e9
    stream = torch.cuda.current_stream()

    # e2e: one kvq_decode_step_host call per step -- the new query and the new
    # token's K/V from pinned host memory, append (quantise-on-write at
    # position seq_len - 1), decode, output back to pinned host memory
    pin = lambda t: t.pin_memory()
    h_q = pin(torch.from_numpy(np.ascontiguousarray(inp.q).view(np.int16)).view(torch.bfloat16))
    last = Tcap - 1
    h_k = pin(torch.from_numpy(np.ascontiguousarray(inp.k[:, :, last]).view(np.int16)).view(torch.bfloat16))
    h_v = pin(torch.from_numpy(np.ascontiguousarray(inp.v[:, :, last]).view(np.int16)).view(torch.bfloat16))
    h_out = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    e2e_ok = bool(np.all(inp.seq_lens == Tcap))
    step_call = kvq.DecodeStepHost(h_q, h_k, h_v, sl, h_out, inp.softmax_scale, out_dtype=kvq.OUT_BF16,
                                   workspace=ws, stream=stream, device=dev)

    def e2e_step(i):
        kc_i, vc_i = caches[i % n_copies]
        step_call.run(kc_i, vc_i)

    e2e = None
    if e2e_ok:
        # at least two calls per cache pair before timing: the library replays
        # a repeated step from a graph captured on its second call
        for i in range(max(args.warmup, 2 * n_copies)):
            e2e_step(i)
        torch.cuda.synchronize()
        et = []
        for i in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_step(i)
            e1.record(stream)
            e1.synchronize()          # the step's result is read back before the next step
            et.append(e0.elapsed_time(e1) / 1e3)
        te = max_over_ranks(torch, dist, sum(et), dev)
        e2e = {"value": job_gbs(bytes_per_step, world, args.steps, te), "unit": "GB/s",
               "h2d_bytes_per_step": int(h_q.numel() * 2 + h_k.numel() * 2 + h_v.numel() * 2),
               "d2h_bytes_per_step": int(h_out.numel() * 2),
               "ms_per_step": te / args.steps * 1e3,
               "us_median": statistics.median(et) * 1e6, "us_p95": _p95(et) * 1e6,
               "step": "one kvq_decode_step_host call from pinned host buffers: the append launch reads the "
                       "new K/V rows and q over the host link (quantise-on-write of K and V, q staged), the decode "
                       "launch writes the bf16 output into host memory; a repeated step's two launches are "
                       "replayed by the library from a CUDA graph captured on its second call"}

    del caches, d
    torch.cuda.empty_cache()
    quant = None
    if rank == 0:
        quant = bench_quantize(torch, kvq, inp, peaks, max(5, min(args.steps, 20)), 3, dev)
    head_bits = None
    if rank == 0:
        head_bits = bench_head_bits(torch, kvq, W, peaks, max(5, min(args.steps, 20)), 3, dev)
    prefill = None
    if not args.no_prefill and rank == 0:
        prefill = bench_prefill(torch, kvq, W, peaks, max(3, min(args.steps, 10)), 3, dev)
        prefill["non_causal"] = bench_prefill(torch, kvq, W, peaks, 3, 3, dev, causal=False)
        prefill["varlen"] = bench_prefill_varlen(torch, kvq, W, peaks, 5, 3, dev)
    extras = None
    if not args.no_extras and rank == 0:
        extras = bench_extra_decodes(torch, kvq, W, peaks, dev, args.steps, args.warmup)
    phase = None
    if not args.no_extras and not args.no_prefill and rank == 0:
        phase = bench_phase_policy(torch, kvq, W, peaks, max(3, min(args.steps, 10)), 3, dev, decode_policy)

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        # every host core (one oracle process each), and one core alone
        cpu = _cpu_entry(_oracle_subprocess(args.workload, 15.0, procs=0))
        cpu["single_core"] = _cpu_entry(_oracle_subprocess(args.workload, 10.0))
        if prefill is not None and "unavailable" not in prefill:
            prefill["cpu_baseline"] = _cpu_entry(_oracle_subprocess("prefill_causal", 10.0))

    if rank == 0:
        traffic = _traffic_from_profile("kvq_decode.cu", args.workload)
        line = {
            "metric": METRIC,
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": avg * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u8/u4 codes, f16 mma, f32 accumulate", "data": "synthetic (seeded, kvq_workloads)",
            "config": {"workload": inp.name, "B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "context": int(Tcap),
                       "bits": [int(b) for b in inp.head_bits],
                       "l2": f"inputs larger than L2: {n_copies} cache copies ({n_copies * bytes_per_step / 1e6:.0f} MB) "
                             "visited in turn, steps back to back",
                       "per_rank": "each rank decodes its own batch (independent sequences)",
                       "timing": timing},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "kernel": "decode_split_kernel (one launch per step, merge fused)",
                         "algorithmic_bytes_per_launch": bytes_per_step, "peak_src": peaks["hbm_src"]},
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clk.summary(),
            "gpu_launches": args.steps,
            "quantize": quant,
            "prefill": prefill,
            "head_bits": head_bits,
            "other_decode_workloads": extras,
            "phase_policy": phase,
            "decode_isolated_launch_us": isolated_us,
            "decode_isolated_device_us": isolated_dev_us,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
