"""The GPU-vs-oracle comparison (tests/parity.py) checked on the CPU.

The oracle's float64 mode is a second correct implementation of the step (it
rounds at the same BF16 points but computes everything else in double), so
`compare` must accept its results in place of the GPU's; results with a
planted deviation must be rejected."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from linear_attention_recurrent_kda_gb300.workloads import Workload, make_inputs
from tests.hostdata import to_oracle
from tests.parity import compare


def fake_gpu(inp):
    o = to_oracle(inp)
    r = oracle.run(o, mode="f64", want_intermediates=True)
    res = {"output": r["output"], "state": r["state"], "conv_state": r["conv_state"],
           "err": r["err"], "dbg": r["inter"]}
    if o["record"]:
        res["rec_u"], res["rec_kg"] = r["rec_u"], r["rec_kg"]
    return res


def wl(**kw):
    base = dict(name="m", batch=6, heads=3, tokens=1, num_slots=16, conv_width=3,
                slot_layout="decode", pad=1, seed=77)
    base.update(kw)
    return Workload(**base)


@pytest.mark.parametrize("w", [wl(), wl(tokens=3, slot_layout="verify", conv_width=5,
                                        num_slots=20, gate_mode=1, has_bias=True),
                               wl(tokens=4, slot_layout="checkpoint", conv_width=6,
                                  record=True)])
def test_second_implementation_passes(w):
    inp = make_inputs(w)
    compare(inp, fake_gpu(inp))
    items = np.array([0, 4, 7, 11, 17])
    compare(inp, fake_gpu(inp), items=items)


@pytest.mark.parametrize("plant", ["state", "output", "conv", "dbg", "pad", "err"])
def test_planted_deviation_fails(plant):
    w = wl(tokens=2, slot_layout="verify", conv_width=4, num_slots=20)
    inp = make_inputs(w)
    g = fake_gpu(inp)
    o = to_oracle(inp)
    r = 0 if o["slots"][0, int(o["accepted"][0]) - 1] > 0 else 1
    if plant == "state":
        s = int(o["slots"][r, 0])
        g["state"][s, 0, 3, 5] += 1e-3
    elif plant == "output":
        g["output"][r * 2, 7] ^= 0x0004       # a few ulps
    elif plant == "conv":
        s = int(o["slots"][r, 0])
        g["conv_state"][s, 0, 1] ^= 0x0001
    elif plant == "dbg":
        g["dbg"][r, 0, 0, 1, 3] ^= 0x0002
    elif plant == "pad":
        pr = [q for q in range(w.batch) if o["slots"][q, int(o["accepted"][q]) - 1] <= 0][0]
        g["output"][pr * 2, 0] = 0x3F80
    elif plant == "err":
        g["err"] = 1
    with pytest.raises(AssertionError):
        compare(inp, g)
