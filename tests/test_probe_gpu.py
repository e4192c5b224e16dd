"""The access-pattern probe (kda_probe_page_copy) on the GPU: every live page
is read and written back in place, so the pool is bit-identical afterwards;
padding slots are skipped, slots beyond the pool raise KDA_DEVERR_SLOT and
are skipped too."""
from __future__ import annotations

import pytest
import torch

from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.api import kda_probe_page_copy
from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int32)


@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("name", ["decode_b64_h32_pad8", "decode_b256_h32", "decode_b4_h8"])
def test_pool_unchanged(name, stages):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    state = inp["state"].cuda()
    before = state.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_probe_page_copy(state=state, slots=inp["slots"].cuda(), stages=stages, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(_bits(state), _bits(before))


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
