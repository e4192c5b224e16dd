"""FP32 conv-state pools (kda_args.conv_f32) on both kernel paths.

* oracle parity (anchored comparison) with FP32 taps that are not BF16 values;
* an FP32 pool holding BF16 values gives the same bits as the BF16 pool.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.workloads import Workload, make_inputs
from tests.parity import compare, run_gpu

pytestmark = pytest.mark.gpu

CASES = {
    "decode": dict(tokens=1, slot_layout="decode", conv_width=3),
    "verify4": dict(tokens=4, slot_layout="verify", conv_width=7, has_bias=True),
    "record8": dict(tokens=8, slot_layout="checkpoint", conv_width=10, record=True,
                    gate_mode=1),
}


def wl(name, **kw):
    c = dict(CASES[name])
    T = c["tokens"]
    base = dict(name="c32_" + name, batch=30, heads=5, num_slots=30 * T + 9, pad=3,
                seed=500 + T, conv_dtype="f32")
    base.update(c)
    base.update(kw)
    return Workload(**base)


@pytest.mark.parametrize("path", [kl.KDA_PATH_PERSISTENT, kl.KDA_PATH_SPLIT])
@pytest.mark.parametrize("name", list(CASES))
def test_fp32_conv_pool_oracle_parity(name, path):
    inp = make_inputs(wl(name))
    assert inp["conv_state"].dtype == torch.float32
    compare(inp, run_gpu(inp, path=path))


@pytest.mark.parametrize("name", list(CASES))
def test_fp32_pool_of_bf16_values_equals_bf16_pool(name):
    inp = make_inputs(wl(name, conv_dtype="bf16"))
    a = run_gpu(inp, path=kl.KDA_PATH_PERSISTENT)
    inp32 = dict(inp, conv_state=inp["conv_state"].float())
    b = run_gpu(inp32, path=kl.KDA_PATH_PERSISTENT)
    for key in ("output", "state", "dbg", "rec_u", "rec_kg"):
        if key in a:
            assert np.array_equal(np.asarray(a[key]).view(np.uint8),
                                  np.asarray(b[key]).view(np.uint8)), key
    conv_a = torch.from_numpy(a["conv_state"].view(np.int16)).view(torch.bfloat16).float()
    assert torch.equal(conv_a, torch.from_numpy(b["conv_state"]))
