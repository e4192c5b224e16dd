"""The N>1 host-side path of bench.py on CPU: world size 2 over gloo.

Each rank runs its own independent batch (weak scaling); the only
collectives are timing reductions (max over ranks).  These tests run the
reduction helper in a real 2-process gloo group, check the per-rank shards,
and launch the reference arm under torchrun with two processes."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank], dist, "cpu")
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r] == [2.0, 10.0, 0.5]


def test_rank_shards_are_independent_batches():
    sys.path.insert(0, ROOT)
    import bench
    from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS["decode_b4_h8"]
    a, b = bench.shard_workload(w, 0), bench.shard_workload(w, 1)
    assert (a.batch, a.heads, a.tokens) == (b.batch, b.heads, b.tokens)
    assert a.seed != b.seed and a == w
    xa, xb = make_inputs(a)["x"], make_inputs(b)["x"]
    assert xa.shape == xb.shape and not torch.equal(xa, xb)


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
           "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--workload", "decode_b4_h8"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_counts_only_the_items_it_runs():
    """The reference arm's sample is capped at the workload's items, so a
    small workload's rate counts the items the oracle actually stepped."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS
    args = argparse.Namespace(steps=1, warmup=0, gpus=1, oracle_threads=1)
    line = bench.run_reference(args, WORKLOADS["decode_b4_h8"])
    assert line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["sample"].startswith("32 of 32 items")
    # value = items stepped / time of a step, and ms_per_step the whole workload
    assert abs(line["value"] * line["ms_per_step"] * 1e-3 - 32) < 1e-6 * 32
