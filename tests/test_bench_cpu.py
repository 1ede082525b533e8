"""Host-side logic of bench.py on CPU: the reference (oracle) arm's JSON
line, and the multi-rank path (independent per-rank batches, max-over-ranks
timing) as world-size-2 gloo ranks."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, check=True,
                         cwd=ROOT)
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 3 and d["value"] > 0
    assert d["unit"] == bench.UNIT and d["metric"] == bench.METRIC
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = bench.make_case("bs4_t8_bf16", seed=bench.rank_seed(rank))
        local_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        m = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        from gated_deltanet_linear_sm_gb300 import synth
        q.put((rank, m, int(case.q[:4].astype(np.int64).sum()), synth.token_head_updates(case)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo_max_timing_and_independent_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, h0, u0), (r1, m1, h1, u1) = res
    assert m0 == m1 == 15.0                              # both see the slowest rank
    assert h0 != h1                                      # each rank has its own batch
    assert u0 == u1
    v = bench.whole_job_value(u0, 2, m0, steps=100)
    assert v == pytest.approx(2 * u0 / (15.0e-3 / 100))
