"""The bench's multi-rank logic on CPU: two gloo ranks (127.0.0.1) must agree
on the slowest rank's time, the whole-job throughput counts every rank's
bytes, and the reference arm runs on rank 0 only."""
import importlib.util
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        local = [0.031, 0.047][rank]            # each rank's own step time
        t = b.max_over_ranks(torch, dist, local, "cpu")
        out[rank] = (t, b.job_gbs(150_994_944, world, 20, t))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    t, gbs = res[0]
    assert t == pytest.approx(0.047)
    assert gbs == pytest.approx(150_994_944 * 2 * 20 / 0.047 / 1e9)


def test_single_rank_helpers_without_a_process_group():
    b = _bench()
    assert b.max_over_ranks(torch, None, 0.5, "cpu") == 0.5
    assert b.job_gbs(1_000_000_000, 1, 10, 2.0) == pytest.approx(5.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    b = _bench()

    class Args:
        workload = "decode_gqa"
        steps = 1
        warmup = 0

    b.run_reference(Args(), 1)    # any rank but 0 returns without work or output
    assert capsys.readouterr().out == ""


def test_reference_arm_line_pairs_with_the_main_arm(capsys, monkeypatch):
    """The reference arm prints the main arm's metric, unit and direction (so
    the two lines can be paired), its oracle run on a pool of worker
    processes, and a prefill sub-object."""
    import json
    b = _bench()
    monkeypatch.setattr(b.os, "cpu_count", lambda: 2)
    monkeypatch.setattr(b, "_oracle_subprocess", lambda w, s, procs=1: {
        "value": 1e-6, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": "stub"})

    class Args:
        workload = "decode_tiny"
        steps = 2
        warmup = 0
        gpus = 1
        step_seconds = 0.2

    b.run_reference(Args(), 0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == b.METRIC
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["cores"] == 2 and line["value"] > 0
    assert line["prefill"]["unit"] == "TFLOP/s"
