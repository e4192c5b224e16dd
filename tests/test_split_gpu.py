"""The cluster-split path (one item over 4 CTAs, path = 2) of the KDA step.

* parity with the oracle (anchored comparison) on decode, verify, record,
  gate_mode 1 + bias, padding and error items;
* the split path and the persistent path (path = 1) give the same bits for
  every output: pools, outputs, records, the BF16 intermediates, the error word.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, Workload, make_inputs
from tests.parity import compare, run_gpu

pytestmark = pytest.mark.gpu

CASES = {
    "decode": dict(tokens=1, slot_layout="decode", conv_width=3),
    "decode_gm1_bias": dict(tokens=1, slot_layout="decode", conv_width=3, gate_mode=1,
                            has_bias=True),
    "verify3": dict(tokens=3, slot_layout="verify", conv_width=6),
    "verify8": dict(tokens=8, slot_layout="verify", conv_width=10),
    "record4": dict(tokens=4, slot_layout="checkpoint", conv_width=6, record=True,
                    gate_mode=1, has_bias=True),
    "record8": dict(tokens=8, slot_layout="checkpoint", conv_width=10, record=True),
}


def wl(name):
    kw = dict(CASES[name])
    T = kw["tokens"]
    base = dict(name="split_" + name, batch=9, heads=5, num_slots=9 * T + 12, pad=2,
                seed=400 + T + 10 * int(kw.get("record", False)))
    base.update(kw)
    return Workload(**base)


@pytest.mark.parametrize("name", list(CASES))
def test_split_path_oracle_parity(name):
    inp = make_inputs(wl(name))
    compare(inp, run_gpu(inp, path=kl.KDA_PATH_SPLIT))


@pytest.mark.parametrize("name", list(CASES))
def test_split_and_persistent_paths_agree_bitwise(name):
    inp = make_inputs(wl(name))
    a = run_gpu(inp, path=kl.KDA_PATH_PERSISTENT)
    b = run_gpu(inp, path=kl.KDA_PATH_SPLIT)
    for key in ("output", "state", "conv_state", "dbg", "rec_u", "rec_kg"):
        if key in a:
            x, y = np.asarray(a[key]), np.asarray(b[key])
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), key
    assert a["err"] == b["err"]


def test_split_error_items():
    T = 3
    w = Workload("split_err", batch=6, heads=4, tokens=T, num_slots=6 * T + 1,
                 conv_width=T + 2, slot_layout="verify", pad=0, seed=77)
    inp = make_inputs(w)
    inp["slots"][1, 1] = 10_000
    inp["accepted"][2] = 0
    inp["slots"][4, 0] = -1
    inp["accepted"][4] = 2
    a = run_gpu(inp, path=kl.KDA_PATH_SPLIT)
    assert a["err"] == kl.KDA_DEVERR_SLOT | kl.KDA_DEVERR_ACCEPTED
    compare(inp, a)


def test_automatic_path_small_batch_uses_split_bits():
    inp = make_inputs(WORKLOADS["decode_b4_h8"])
    a = run_gpu(inp, path=kl.KDA_PATH_AUTO)
    b = run_gpu(inp, path=kl.KDA_PATH_SPLIT)
    assert np.array_equal(a["output"], b["output"])
    assert np.array_equal(a["state"].view(np.uint32), b["state"].view(np.uint32))
