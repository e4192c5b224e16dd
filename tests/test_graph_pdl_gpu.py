"""Chaining the KDA step: CUDA-graph replay and programmatic dependent launch.

* A decode step captured once in a CUDA graph and replayed three times gives
  the same pools and outputs, bit for bit, as three eager steps.
* With use_pdl the kernel may start before the preceding kernel ends; its
  producer waits (griddepcontrol) before reading the step inputs that kernel
  writes, so a predecessor that writes x gives the same result as without PDL.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_attention_recurrent_kda_gb300.api import step_from_inputs
from linear_attention_recurrent_kda_gb300.workloads import Workload, make_inputs
from tests.parity import to_device

pytestmark = pytest.mark.gpu


def wl(**kw):
    base = dict(name="g", batch=48, heads=7, tokens=1, num_slots=80, conv_width=3,
                slot_layout="decode", pad=4, seed=321)
    base.update(kw)
    return Workload(**base)


def snapshot(d, out):
    torch.cuda.synchronize()
    return [d["state"].clone(), d["conv_state"].clone(), out.clone()]


@pytest.mark.parametrize("tokens", [1, 3])
def test_cuda_graph_replay_equals_eager(tokens):
    w = wl(tokens=tokens, slot_layout="decode" if tokens == 1 else "verify",
           conv_width=tokens + 2, num_slots=48 * tokens + 9)
    inp = make_inputs(w)
    B, H = w.batch, w.heads
    de, dg = to_device(inp), to_device(inp)
    oe = torch.zeros((B * tokens, H * 128), dtype=torch.bfloat16, device="cuda")
    og = torch.zeros_like(oe)
    se = step_from_inputs(de, oe)
    sg = step_from_inputs(dg, og)
    # one eager call on a throwaway copy configures the kernel before capture
    dw = to_device(inp)
    step_from_inputs(dw, torch.zeros_like(oe))()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        sg()
    for _ in range(3):
        se()
        graph.replay()
    a, b = snapshot(de, oe), snapshot(dg, og)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_pdl_after_a_kernel_that_writes_x():
    w = wl()
    inp = make_inputs(w)
    B, H = w.batch, w.heads
    x_new = torch.randn(inp["x"].shape, generator=torch.Generator().manual_seed(9))
    x_new = x_new.to(torch.bfloat16).cuda()
    outs = []
    for pdl in (False, True):
        d = to_device(inp)
        out = torch.zeros((B, H * 128), dtype=torch.bfloat16, device="cuda")
        st = step_from_inputs(d, out, use_pdl=pdl)
        torch.cuda.synchronize()
        torch.add(x_new, 0, out=d["x"])      # predecessor kernel writes x
        st()
        outs.append(snapshot(d, out))
    for x, y in zip(*outs):
        assert torch.equal(x, y)
