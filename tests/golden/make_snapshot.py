"""Writes ``oracle_snapshot.json``: the oracle's results on three small
seeded steps (a decode, a verify and a record-mode verify) and two small
output-projection consumer calls, in both of the oracle's modes.  The pages print no worked example with values, so nothing here is
a value from the pages: this file freezes the oracle itself, so that any
later change to its arithmetic shows up in ``tests/test_golden.py`` and has
to be justified by the passage it follows.  It calls only ``oracle/`` and
the seeded input generator.

    python tests/golden/make_snapshot.py
"""
from __future__ import annotations

import dataclasses
import hashlib
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from linear_attention_recurrent_kda_gb300.workloads import (OprojWorkload, Workload,  # noqa: E402
                                                            make_oproj_inputs, make_inputs)
from tests.hostdata import to_oracle  # noqa: E402

CASES = [
    Workload("snap_decode", batch=3, heads=2, tokens=1, num_slots=8, conv_width=3,
             slot_layout="decode", pad=1, seed=7001),
    Workload("snap_verify", batch=2, heads=2, tokens=3, num_slots=2 * 3 + 3, conv_width=5,
             slot_layout="verify", gate_mode=1, has_bias=True, seed=7002),
    Workload("snap_record", batch=2, heads=1, tokens=4, num_slots=4, conv_width=6,
             slot_layout="checkpoint", record=True, seed=7003),
]
OPROJ_CASES = [
    OprojWorkload("snap_oproj", tp=5, tokens=3, hidden=512, nb=3, has_delta=True, seed=7011),
    OprojWorkload("snap_oproj_plain", tp=2, tokens=2, hidden=256, nb=0, has_delta=False,
                  seed=7012),
]
SAMPLES = 32          # sampled elements per written page / record array


def sample_index(n: int, seed: int) -> np.ndarray:
    return np.sort(np.random.default_rng(seed).choice(n, size=min(SAMPLES, n), replace=False))


def snapshot(w: Workload, mode: str) -> dict:
    o = to_oracle(make_inputs(w))
    res = oracle.run(o, mode=mode)
    state0 = np.asarray(o["state"])
    changed = [int(s) for s in range(w.num_slots)
               if not np.array_equal(res["state"][s].view(np.uint32), state0[s].view(np.uint32))]
    pages = {}
    for s in changed:
        flat = res["state"][s].reshape(-1)
        idx = sample_index(flat.size, 100 + s)
        pages[str(s)] = {"index": idx.tolist(), "value": [float(v) for v in flat[idx]]}
    out = {"output_bf16_hex": res["output"].reshape(-1).view(np.uint16).tobytes().hex(),
           "conv_state_sha256": hashlib.sha256(
               np.ascontiguousarray(res["conv_state"]).tobytes()).hexdigest(),
           "pages_written": changed, "pages": pages, "err": res["err"]}
    if w.record:
        flat = res["rec_u"].reshape(-1)
        idx = sample_index(flat.size, 99)
        out["rec_u"] = {"index": idx.tolist(), "value": [float(v) for v in flat[idx]]}
        out["rec_kg_hex"] = res["rec_kg"].reshape(-1).view(np.uint16).tobytes().hex()
    return out


def oproj_bits(t):
    return None if t is None else t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oproj_snapshot(w: OprojWorkload, mode: str) -> dict:
    h = make_oproj_inputs(w)
    res = oracle.oproj(partials=oproj_bits(h["partials"]), prefix=oproj_bits(h["prefix"]),
                       out_norm=oproj_bits(h["out_norm"]), blocks=oproj_bits(h["blocks"]),
                       norm=oproj_bits(h["norm"]), query=oproj_bits(h["query"]),
                       has_delta=h["has_delta"], eps=h["eps"], out_eps=h["out_eps"], mode=mode)
    return {"prefix_bf16_sha256": hashlib.sha256(res["prefix"].tobytes()).hexdigest(),
            "output_bf16_sha256": hashlib.sha256(res["output"].tobytes()).hexdigest(),
            "output_bf16_head_hex": res["output"].reshape(-1)[:16].tobytes().hex()}


def main() -> None:
    doc = {"about": "oracle snapshot on small seeded steps; regenerate with "
                    "tests/golden/make_snapshot.py after a justified oracle change",
           "cases": []}
    for w in CASES:
        doc["cases"].append({"workload": dataclasses.asdict(w),
                             "f32": snapshot(w, "f32"), "f64": snapshot(w, "f64")})
    doc["oproj_cases"] = [{"workload": dataclasses.asdict(w), "f32": oproj_snapshot(w, "f32"),
                           "f64": oproj_snapshot(w, "f64")} for w in OPROJ_CASES]
    with open(os.path.join(HERE, "oracle_snapshot.json"), "w") as f:
        json.dump(doc, f, separators=(",", ":"))
        f.write("\n")


if __name__ == "__main__":
    main()
