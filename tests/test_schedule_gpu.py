"""The persistent kernel's item schedule: contiguous ranges, then shared items.

With scheduler words (kda_args.sched) each CTA walks a contiguous range (7/8
of its even share for decode with many items per CTA and for record steps,
else all but the remainder of an even split) and the remaining items go one
at a time to whichever CTA asks first; without them every item sits in a
fixed contiguous range.  Items are
independent, so both must give the same bits on every output, pool, record
and the error word, and the words must be back at zero after every launch
(the last CTA zeroes them).  The oracle comparisons of the other GPU tests
run with the binding's default words; these tests pin the schedule itself,
and kda_step_noalloc, the same step on the library's own static words.
"""
from __future__ import annotations

import pytest
import torch

from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.api import step_from_inputs
from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, Workload, make_inputs
from tests.hostdata import bits
from tests.parity import compare, run_gpu, same_bits, to_device

pytestmark = pytest.mark.gpu


def wl(**kw) -> Workload:
    base = dict(name="s", batch=61, heads=5, tokens=1, num_slots=96, conv_width=3,
                slot_layout="decode", pad=7, seed=611)
    base.update(kw)
    return Workload(**base)


CASES = [WORKLOADS[n] for n in sorted(WORKLOADS)] + [
    # 305 items: one static item per CTA, the other 153 shared
    wl(),
    # 160 items (just over one per SM): no static items at all
    wl(batch=32, heads=5, seed=612, pad=3),
    # verify and record, padded rows among the shared items
    wl(batch=70, heads=4, tokens=3, num_slots=3 * 70 + 1, conv_width=5,
       slot_layout="verify", pad=9, seed=613),
    wl(batch=50, heads=6, tokens=5, num_slots=51, conv_width=8,
       slot_layout="checkpoint", record=True, pad=4, seed=614, gate_mode=1),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name + f"_t{c.tokens}" for c in CASES])
def test_shared_items_same_bits_as_fixed_ranges(w):
    inp = make_inputs(w)
    fixed = run_gpu(inp, dbg=False, balance=False, path=kl.KDA_PATH_PERSISTENT)
    shared = run_gpu(inp, dbg=False, balance=True, path=kl.KDA_PATH_PERSISTENT)
    same_bits(shared, fixed)


def _launch(w, sched, use_pdl=False, dbg=False):
    d = to_device(make_inputs(w))
    B, H, T = d["batch"], d["heads"], d["tokens"]
    out = torch.full((B * T, H * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    dbgt = (torch.zeros((B, H, T, 4, 128), dtype=torch.bfloat16, device="cuda")
            if dbg else None)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ru = rk = None
    if d["record"]:
        ru = torch.zeros((B, H, T, 128), dtype=torch.float32, device="cuda")
        rk = torch.zeros((B, H, T, 256), dtype=torch.bfloat16, device="cuda")
    step = step_from_inputs(d, out, rec_u=ru, rec_kg=rk, err=err, sched=sched,
                            use_pdl=use_pdl, path=kl.KDA_PATH_PERSISTENT, dbg=dbgt)
    step.dbg_buf = dbgt
    return d, out, err, ru, rk, step


def test_words_return_to_zero_and_repeat_bits():
    """Twenty launches on one pair of words, pools restored before each: every
    launch reproduces the first one's bits and leaves the words at zero."""
    w = WORKLOADS["verify_q8_record_b64_h64"]
    sched = torch.zeros(2, dtype=torch.int32, device="cuda")
    d, out, err, ru, rk, step = _launch(w, sched)
    st0, cv0 = d["state"].clone(), d["conv_state"].clone()
    ref = None
    for i in range(20):
        d["state"].copy_(st0)
        d["conv_state"].copy_(cv0)
        out.fill_(float("nan"))
        ru.fill_(float("nan"))
        step()
        torch.cuda.synchronize()
        assert sched.tolist() == [0, 0], f"launch {i} left {sched.tolist()}"
        cur = [out.clone(), d["state"].clone(), d["conv_state"].clone(), ru.clone(), rk.clone()]
        if ref is None:
            ref = cur
            continue
        for a, b in zip(cur, ref):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert int(err.item()) == 0


def test_steps_sharing_words_on_one_stream_and_pdl():
    """Two decode steps on disjoint pools share one pair of words, the second
    launched with PDL right behind the first (its shared items are asked for
    only after the wait, when the first has zeroed the words): each matches
    the oracle, and the words end at zero."""
    sched = torch.zeros(2, dtype=torch.int32, device="cuda")
    wa, wb = wl(seed=615), wl(seed=616, batch=57)
    la = _launch(wa, sched, dbg=True)
    lb = _launch(wb, sched, use_pdl=True, dbg=True)
    la[5]()
    lb[5]()
    torch.cuda.synchronize()
    assert sched.tolist() == [0, 0]
    for w, (d, out, err, _, _, step) in ((wa, la), (wb, lb)):
        gpu = {"output": bits(out), "state": d["state"].cpu().numpy(),
               "conv_state": bits(d["conv_state"]), "err": int(err.item()),
               "dbg": bits(step.dbg_buf)}
        compare(make_inputs(w), gpu)


def test_graph_replays_share_words():
    """A step captured once and replayed five times: each replay equals an
    eager launch from the same pools, and the words end at zero."""
    w = wl(seed=617, batch=90)
    sched = torch.zeros(2, dtype=torch.int32, device="cuda")
    d, out, err, ru, rk, step = _launch(w, sched)
    st0, cv0 = d["state"].clone(), d["conv_state"].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    torch.cuda.synchronize()
    d["state"].copy_(st0)
    d["conv_state"].copy_(cv0)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    got = [out.clone(), d["state"].clone(), d["conv_state"].clone()]
    assert sched.tolist() == [0, 0]
    d["state"].copy_(st0)
    d["conv_state"].copy_(cv0)
    for _ in range(5):
        step()
    torch.cuda.synchronize()
    for a, b in zip(got, [out, d["state"], d["conv_state"]]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert int(err.item()) == 0


@pytest.mark.parametrize("w", CASES, ids=[c.name + f"_t{c.tokens}" for c in CASES])
def test_noalloc_entry_same_bits(w):
    """kda_step_noalloc (the library's own words) gives the fixed-range bits,
    twice in a row (the first launch left the words at zero)."""
    inp = make_inputs(w)
    fixed = run_gpu(inp, dbg=False, balance=False, path=kl.KDA_PATH_PERSISTENT)
    for _ in range(2):
        own = run_gpu(inp, dbg=False, noalloc=True, path=kl.KDA_PATH_PERSISTENT)
        same_bits(own, fixed)


def test_noalloc_entry_repeated_launches_and_oracle():
    """Thirty launches through kda_step_noalloc on one stream, pools restored
    before each, reproduce the first launch's bits; one more from the seeded
    pools matches the oracle (its items all ran: a word left non-zero would
    hand out no shared items)."""
    w = wl(seed=618, batch=200, heads=6, num_slots=256, pad=11)
    d = to_device(make_inputs(w))
    B, H, T = d["batch"], d["heads"], d["tokens"]
    out = torch.full((B * T, H * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dbgt = torch.zeros((B, H, T, 4, 128), dtype=torch.bfloat16, device="cuda")
    step = step_from_inputs(d, out, err=err, dbg=dbgt, noalloc=True,
                            path=kl.KDA_PATH_PERSISTENT)
    st0, cv0 = d["state"].clone(), d["conv_state"].clone()
    ref = None
    for _ in range(30):
        d["state"].copy_(st0)
        d["conv_state"].copy_(cv0)
        out.fill_(float("nan"))
        step()
        cur = [out.clone(), d["state"].clone(), d["conv_state"].clone()]
        if ref is None:
            ref = cur
        else:
            for a, b in zip(cur, ref):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    torch.cuda.synchronize()
    gpu = {"output": bits(out), "state": d["state"].cpu().numpy(),
           "conv_state": bits(d["conv_state"]), "err": int(err.item()), "dbg": bits(dbgt)}
    compare(make_inputs(w), gpu)
