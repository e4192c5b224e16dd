"""Host threads calling the library at once, from its first call on.

A fresh process (the library's per-device set-up not yet done) prepares
eight steps of different kinds -- decode, verify, record, on the persistent
and the cluster-split paths -- and releases eight host threads together, each
launching its step on its own stream (ctypes drops the GIL for the call, so
the first-call set-up of every kernel really runs concurrently).  Every
result must pass the anchored comparison with the oracle.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, threading
import torch
from linear_attention_recurrent_kda_gb300.api import step_from_inputs
from linear_attention_recurrent_kda_gb300.workloads import Workload, make_inputs
from tests.hostdata import bits
from tests.parity import compare, to_device

cases = [
    dict(tokens=1, slot_layout="decode", conv_width=3, path=1),
    dict(tokens=1, slot_layout="decode", conv_width=3, path=2),
    dict(tokens=3, slot_layout="verify", conv_width=5, path=1),
    dict(tokens=3, slot_layout="verify", conv_width=5, path=2),
    dict(tokens=4, slot_layout="checkpoint", conv_width=6, record=True, path=1),
    dict(tokens=8, slot_layout="checkpoint", conv_width=10, record=True, path=1),
    dict(tokens=2, slot_layout="verify", conv_width=4, gate_mode=1, has_bias=True, path=1),
    dict(tokens=1, slot_layout="decode", conv_width=3, gate_mode=1, has_bias=True, path=1),
]
jobs = []
for n, kw in enumerate(cases):
    path = kw.pop("path")
    T = kw["tokens"]
    w = Workload(name=f"thr{n}", batch=12 + n, heads=5, num_slots=(12 + n) * T + 4,
                 pad=2, seed=700 + n, **kw)
    inp = make_inputs(w)
    d = to_device(inp)
    B, H = w.batch, w.heads
    out = torch.full((B * T, H * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    rec_u = rec_kg = None
    if w.record:
        rec_u = torch.zeros((B, H, T, 128), dtype=torch.float32, device="cuda")
        rec_kg = torch.zeros((B, H, T, 256), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dbg = torch.zeros((B, H, T, 4, 128), dtype=torch.bfloat16, device="cuda")
    step = step_from_inputs(d, out, rec_u=rec_u, rec_kg=rec_kg, err=err, dbg=dbg, path=path)
    jobs.append((inp, d, out, rec_u, rec_kg, err, dbg, step, torch.cuda.Stream()))
torch.cuda.synchronize()
gate = threading.Barrier(len(jobs))
failures = []

def run(job):
    step, stream = job[7], job[8]
    try:
        gate.wait()
        step(stream)
    except Exception as e:  # reported by the parent
        failures.append(repr(e))

threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
for t in threads:
    t.start()
for t in threads:
    t.join()
torch.cuda.synchronize()
stats = []
for inp, d, out, rec_u, rec_kg, err, dbg, step, stream in jobs:
    gpu = {"output": bits(out), "state": d["state"].cpu().numpy(),
           "conv_state": bits(d["conv_state"]), "err": int(err.item()), "dbg": bits(dbg)}
    if rec_u is not None:
        gpu["rec_u"] = rec_u.cpu().numpy()
        gpu["rec_kg"] = bits(rec_kg)
    st = compare(inp, gpu)
    stats.append(st["out_max_ulp"])
print(json.dumps({"failures": failures, "out_max_ulp": stats}))
"""


def test_concurrent_first_calls_from_host_threads():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    res = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-4000:]
    rep = json.loads(res.stdout.strip().splitlines()[-1])
    assert rep["failures"] == []
    assert len(rep["out_max_ulp"]) == 8
