"""Chaining the KDA step: CUDA-graph replay and programmatic dependent launch,
checked against the oracle.

* A step captured once in a CUDA graph and replayed: the first replay passes
  the anchored comparison against the oracle on the inputs; the third replay
  against the oracle run from the pools the second left; and three replays
  equal three eager steps bit for bit.
* With use_pdl the kernel may start before the preceding kernel ends.  Its
  producer reads only the state pages, slots and accepted before waiting
  (griddepcontrol) on that kernel; every other input is read, and every output
  written, after the wait (KdaWide.kernel: the state rows first, then the
  wait, then x, gate, f_a and beta).  So a predecessor that rewrites x, gate,
  f_a, beta, the norm weight and the conv pool gives the oracle's result on
  the new values; and a step whose gate input is the previous step's output
  (two steps chained by PDL on disjoint pools, the first one triggering its
  dependents early) gives the oracle's result on that output.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_attention_recurrent_kda_gb300.api import step_from_inputs
from linear_attention_recurrent_kda_gb300.workloads import Workload, make_inputs
from tests.hostdata import bits
from tests.parity import compare, to_device

pytestmark = pytest.mark.gpu


def wl(**kw):
    base = dict(name="g", batch=48, heads=7, tokens=1, num_slots=80, conv_width=3,
                slot_layout="decode", pad=4, seed=321)
    base.update(kw)
    return Workload(**base)


class Launch:
    """Device copies of a workload's inputs with output, dbg and error buffers,
    and the prepared step over them."""

    def __init__(self, inp, use_pdl=False, gate=None):
        self.inp = inp
        d = to_device(inp)
        if gate is not None:
            d["gate"] = gate
        B, H, T = d["batch"], d["heads"], d["tokens"]
        self.d = d
        self.out = torch.full((B * T, H * 128), float("nan"), dtype=torch.bfloat16,
                              device="cuda")
        self.dbg = torch.zeros((B, H, T, 4, 128), dtype=torch.bfloat16, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.rec_u = self.rec_kg = None
        if d["record"]:
            self.rec_u = torch.zeros((B, H, T, 128), dtype=torch.float32, device="cuda")
            self.rec_kg = torch.zeros((B, H, T, 256), dtype=torch.bfloat16, device="cuda")
        self.step = step_from_inputs(d, self.out, rec_u=self.rec_u, rec_kg=self.rec_kg,
                                     err=self.err, dbg=self.dbg, use_pdl=use_pdl)

    def pools(self):
        """Host copies of the current pools (inputs of a following step)."""
        torch.cuda.synchronize()
        return self.d["state"].cpu().clone(), self.d["conv_state"].cpu().clone()

    def result(self):
        torch.cuda.synchronize()
        res = {"output": bits(self.out), "state": self.d["state"].cpu().numpy(),
               "conv_state": bits(self.d["conv_state"]), "err": int(self.err.item()),
               "dbg": bits(self.dbg)}
        if self.rec_u is not None:
            res["rec_u"] = self.rec_u.cpu().numpy()
            res["rec_kg"] = bits(self.rec_kg)
        return res

    def snapshot(self):
        torch.cuda.synchronize()
        return [self.d["state"].clone(), self.d["conv_state"].clone(), self.out.clone()]


def layout(tokens, record=False):
    if record:
        return dict(tokens=tokens, slot_layout="checkpoint", conv_width=tokens + 2,
                    record=True, gate_mode=1, has_bias=True, num_slots=60)
    return dict(tokens=tokens, slot_layout="decode" if tokens == 1 else "verify",
                conv_width=tokens + 2, num_slots=48 * tokens + 9)


@pytest.mark.parametrize("tokens,record", [(1, False), (3, False), (4, True)])
def test_cuda_graph_replay_matches_the_oracle(tokens, record):
    w = wl(**layout(tokens, record))
    inp = make_inputs(w)
    eager, graphed = Launch(inp), Launch(inp)
    # one eager call on a throwaway copy configures the kernel before capture
    Launch(inp).step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        graphed.step()
    graph.replay()
    compare(inp, graphed.result())
    graph.replay()
    mid = dict(inp)
    mid["state"], mid["conv_state"] = graphed.pools()
    graph.replay()
    compare(mid, graphed.result())
    for _ in range(3):
        eager.step()
    for x, y in zip(eager.snapshot(), graphed.snapshot()):
        assert torch.equal(x, y)


@pytest.mark.parametrize("tokens,record", [(1, False), (4, False), (4, True)])
def test_pdl_after_a_kernel_that_rewrites_the_inputs(tokens, record):
    w = wl(**layout(tokens, record))
    inp = make_inputs(w)
    g = torch.Generator().manual_seed(9)
    new = dict(inp)
    for key in ("x", "gate", "f_a", "beta", "norm_weight"):
        new[key] = torch.randn(inp[key].shape, generator=g).to(torch.bfloat16)
    new["conv_state"] = torch.randn(inp["conv_state"].shape, generator=g).to(torch.bfloat16)
    for pdl in (False, True):
        L = Launch(inp, use_pdl=pdl)
        staged = {k: new[k].cuda() for k in ("x", "gate", "f_a", "beta", "conv_state",
                                             "norm_weight")}
        torch.cuda.synchronize()
        # predecessor kernels rewrite the inputs the step reads after its wait
        for k, v in staged.items():
            L.d[k].copy_(v)
        L.step()
        compare(new, L.result())


def test_two_steps_chained_by_pdl_on_disjoint_pools():
    """Step B reads, as its output gate, the output step A writes; B is
    launched with PDL right behind A (which triggers its dependents as soon
    as its producers have issued their loads), so B's page loads overlap A
    and B's gate read waits for A to finish."""
    wa = wl(batch=64, heads=8, num_slots=80, pad=5, seed=331)
    wb = wa.with_(seed=332)
    ia, ib = make_inputs(wa), make_inputs(wb)
    A = Launch(ia, use_pdl=True)
    B = Launch(ib, use_pdl=True, gate=A.out)
    torch.cuda.synchronize()
    A.step()
    B.step()
    ra, rb = A.result(), B.result()
    compare(ia, ra)
    ib_seen = dict(ib)
    ib_seen["gate"] = torch.from_numpy(ra["output"].view(np.int16)).view(torch.bfloat16)
    compare(ib_seen, rb)
