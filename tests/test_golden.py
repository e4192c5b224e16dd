"""The oracle against its frozen snapshot (``tests/golden/oracle_snapshot.json``,
written by ``tests/golden/make_snapshot.py`` from the oracle alone).

The pages print no worked example with values, so this is not a pin of the
method (those are in ``test_oracle_pins.py``): it makes any change of the
oracle's results visible.  BF16 outputs, records and conv windows must match
bit for bit; sampled FP32 state and record values to 1e-6 relative (the
oracle's exp and division come from the host's libm, which may differ in
the last bit between hosts)."""
from __future__ import annotations

import hashlib
import json
import os

import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrent_kda_gb300.workloads import (OprojWorkload, Workload,
                                                            make_oproj_inputs, make_inputs)
from tests.hostdata import to_oracle

SNAP = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                    "oracle_snapshot.json")
DOC = json.load(open(SNAP))


def _close(got, want):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    return bool(np.all(np.abs(got - want) <= 1e-6 * np.abs(want) + 1e-30))


@pytest.mark.parametrize("mode", ["f32", "f64"])
@pytest.mark.parametrize("case", range(len(DOC["cases"])))
def test_oracle_matches_snapshot(case, mode):
    c = DOC["cases"][case]
    w = Workload(**c["workload"])
    snap = c[mode]
    o = to_oracle(make_inputs(w))
    res = oracle.run(o, mode=mode)
    assert res["err"] == snap["err"]
    assert res["output"].reshape(-1).view(np.uint16).tobytes().hex() == snap["output_bf16_hex"]
    assert hashlib.sha256(np.ascontiguousarray(res["conv_state"]).tobytes()).hexdigest() == \
        snap["conv_state_sha256"]
    state0 = np.asarray(o["state"])
    changed = [s for s in range(w.num_slots)
               if not np.array_equal(res["state"][s].view(np.uint32), state0[s].view(np.uint32))]
    assert changed == snap["pages_written"]
    for s, pg in snap["pages"].items():
        flat = res["state"][int(s)].reshape(-1)
        assert _close(flat[pg["index"]], pg["value"]), s
    if w.record:
        assert _close(res["rec_u"].reshape(-1)[snap["rec_u"]["index"]], snap["rec_u"]["value"])
        assert res["rec_kg"].reshape(-1).view(np.uint16).tobytes().hex() == snap["rec_kg_hex"]


def _obits(t):
    return None if t is None else t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("mode", ["f32", "f64"])
@pytest.mark.parametrize("case", range(len(DOC["oproj_cases"])))
def test_oproj_oracle_matches_snapshot(case, mode):
    c = DOC["oproj_cases"][case]
    h = make_oproj_inputs(OprojWorkload(**c["workload"]))
    res = oracle.oproj(partials=_obits(h["partials"]), prefix=_obits(h["prefix"]),
                       out_norm=_obits(h["out_norm"]), blocks=_obits(h["blocks"]),
                       norm=_obits(h["norm"]), query=_obits(h["query"]),
                       has_delta=h["has_delta"], eps=h["eps"], out_eps=h["out_eps"], mode=mode)
    assert res["output"].reshape(-1)[:16].tobytes().hex() == c[mode]["output_bf16_head_hex"]
    assert hashlib.sha256(res["prefix"].tobytes()).hexdigest() == c[mode]["prefix_bf16_sha256"]
    assert hashlib.sha256(res["output"].tobytes()).hexdigest() == c[mode]["output_bf16_sha256"]
