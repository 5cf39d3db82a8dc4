"""Host logic of the multi-rank benchmark, run as two gloo ranks on the CPU.

Each rank decodes an independent batch (weak scaling, no data exchange), so
the only cross-rank step is the maximum of the per-rank timings; the job's
throughput is world x per-rank bytes over that maximum.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bit_kv_cache_06_gb300 import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank timings: step, decode, prefill, wall (ms)
        vals = [1.0 + rank, 10.0 - 3.0 * rank, 0.25 * (rank + 1), 7.0]
        got = bench.max_over_ranks(vals, world, torch.device("cpu"))
        queue.put((rank, got))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = [2.0, 10.0, 0.5, 7.0]
    assert results[0] == want and results[1] == want


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 1.5], 1, torch.device("cpu")) == [3.0, 1.5]


def test_whole_job_throughput_is_weak_scaling():
    per_rank = 268599296
    one = bench.whole_job_gbs(1, per_rank, 0.1)
    assert one == pytest.approx(per_rank / 1e-4 / 1e9)
    # eight ranks, each as fast: eight times the bytes in the same time
    assert bench.whole_job_gbs(8, per_rank, 0.1) == pytest.approx(8 * one)


def test_ranks_get_independent_batches():
    w = synth.C1
    k0, v0 = synth.make_kv(w, layer=0)
    k1, v1 = synth.make_kv(w, layer=1)
    assert k0.shape == k1.shape
    assert not torch.equal(k0, k1) and not torch.equal(v0, v1)
    k0b, _ = synth.make_kv(w, layer=0)
    assert torch.equal(k0, k0b)          # seeded: a rank's batch is reproducible


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1"])
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda args: called.append(args) or {})
    bench.main()
    assert called == [] and capsys.readouterr().out == ""


def test_gpus_flag_must_match_world_size(monkeypatch):
    """--gpus N without N ranks (or N ranks without --gpus N) is refused
    before any GPU work: one process drives one GPU."""
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "2", "--steps", "1"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert "WORLD_SIZE" in str(e.value)
