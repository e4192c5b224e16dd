"""The access-pattern probe (kda_probe_page_copy) on the GPU.  Decode: every
live page is read and written back in place, so the pool is bit-identical
afterwards; padding slots are skipped, slots beyond the pool raise
KDA_DEVERR_SLOT and are skipped too.  Verify: each live item's read page
(slot of token accepted-1) lands in the slots of all its tokens, and no
other page changes."""
from __future__ import annotations

import pytest
import torch

from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.probe import kda_probe_page_copy
from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int32)


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("name", ["decode_b64_h32_pad8", "decode_b256_h32", "decode_b4_h8"])
def test_pool_unchanged(name, stages, shared):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    state = inp["state"].cuda()
    before = state.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sched = torch.zeros(2, dtype=torch.int32, device="cuda") if shared else None
    kda_probe_page_copy(state=state, slots=inp["slots"].cuda(), stages=stages, err=err,
                        sched=sched)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(_bits(state), _bits(before))
    if shared:
        assert sched.tolist() == [0, 0]


def test_out_of_pool_slot_flags_and_skips():
    w = WORKLOADS["decode_b4_h8"]
    inp = make_inputs(w)
    slots = inp["slots"].clone()
    slots[1] = w.num_slots          # beyond the pool
    slots[2] = 0                    # padding
    state = inp["state"].cuda()
    before = state.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_probe_page_copy(state=state, slots=slots.cuda(), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kl.KDA_DEVERR_SLOT
    assert torch.equal(_bits(state), _bits(before))


VERIFY = {
    "q4": WORKLOADS["verify_q4_b128_h32"],
    "q8_ragged": Workload("probe_q8", batch=9, heads=4, tokens=8, num_slots=9 * 8 + 5,
                          conv_width=10, slot_layout="verify", pad=2, seed=611),
}


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("name", sorted(VERIFY))
def test_verify_fanout(name, stages, shared):
    w = VERIFY[name]
    inp = make_inputs(w)
    slots, acc, state = inp["slots"], inp["accepted"], inp["state"]
    want = state.clone()
    for r in range(slots.shape[0]):
        src = int(slots[r, int(acc[r]) - 1])
        if src <= 0:
            continue
        for t in range(w.tokens):
            dst = int(slots[r, t])
            if dst > 0:
                want[dst] = state[src]
    g = state.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sched = torch.zeros(2, dtype=torch.int32, device="cuda") if shared else None
    kda_probe_page_copy(state=g, slots=slots.cuda(), accepted=acc.cuda(), tokens=w.tokens,
                        stages=stages, err=err, sched=sched)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(_bits(g.cpu()), _bits(want))
    if shared:
        assert sched.tolist() == [0, 0]


def test_verify_errors_flag_and_skip():
    w = WORKLOADS["verify_q4_b128_h32"]
    inp = make_inputs(w)
    slots, acc = inp["slots"].clone(), inp["accepted"].clone()
    acc[3] = 0                      # accepted out of range
    slots[5, 1] = w.num_slots       # a target beyond the pool
    state = inp["state"]
    g = state.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_probe_page_copy(state=g, slots=slots.cuda(), accepted=acc.cuda(), tokens=w.tokens, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kl.KDA_DEVERR_SLOT | kl.KDA_DEVERR_ACCEPTED
    got = g.cpu()
    for r in (3, 5):                # skipped items wrote nothing
        for t in range(w.tokens):
            s = int(slots[r, t])
            if 0 < s < w.num_slots:
                assert torch.equal(_bits(got[s]), _bits(state[s]))
