"""The bench's multi-rank host logic on CPU: two gloo ranks (world_size 2).

Under torchrun every rank runs its own replica of the layer step (replicas
only: no data-path collective); the job's time is the slowest rank's and its
throughput counts the tokens of all ranks.  The reference arm runs and prints
on rank 0 alone.  These are checked here with the gloo backend; the CUDA
steps in between are the single-GPU path the GPU tests cover."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r's own time is 1 + r seconds: the job's time is the slowest, 2 s
        t = bench.max_over_ranks(1.0 + rank, torch.device("cpu"))
        value = bench.job_tokens_per_s(100, 8, world, t)
        dist.barrier()
        results[rank] = (t, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_tokens():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    assert set(got) == {0, 1}
    for rank in range(world):
        t, value = got[rank]
        assert t == 2.0                       # both ranks agree on the slowest time
        assert value == 100 * 8 * world / 2.0  # tokens of both replicas over that time


def test_single_rank_keeps_its_own_time():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(1.25, torch.device("cpu")) == 1.25
    assert bench.job_tokens_per_s(10, 8, 1, 0.5) == 160.0


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    """The reference arm (the CPU oracle) under torchrun: a rank other than 0
    returns without work and without output."""
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "oracle_steps", lambda *a, **k: called.append(a) or ([1.0], 1, 1, 16))
    args = bench.argparse.Namespace(workload="tiny", warmup=0, steps=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == "" and not called


def test_reference_arm_line_on_rank_zero(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "0")
    # one warm-up step, then two timed whole steps of 16 tokens in 4 s each
    monkeypatch.setattr(bench, "oracle_steps", lambda *a, **k: ([0.5, 4.0, 4.0], 4, 16, 16))
    args = bench.argparse.Namespace(workload="tiny", warmup=1, steps=2)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] == 4.0
    assert res["ms_per_step"] == 4000.0          # the measured whole-step time, not an extrapolation
    assert res["cpu_baseline"]["cores"] == 4 and res["cpu_baseline"]["value"] == 4.0
    assert res["e2e"] == {"value": 4.0, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_steps_split_tokens_over_processes():
    """The CPU arms' runner: whole steps of the tiny layer, its 16 tokens split
    over up to one spawned process per host core; one time per step."""
    times, procs, cores, ntok = bench.oracle_steps("tiny", 2)
    assert ntok == 16 and len(times) == 2 and all(t > 0 for t in times)
    assert procs == min(cores, 16) and cores == len(os.sched_getaffinity(0))
