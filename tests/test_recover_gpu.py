"""GPU tests of the record replay (kda_recover) through the C ABI.

* parity with the oracle's replay on the GPU's own records (exact inputs);
* record-mode verify followed by replay reproduces, bit for bit, the pages a
  non-record verify writes, and record mode's outputs equal the non-record
  outputs bit for bit (both on the GPU: same operations);
* padding, error rows and accepted = 0 (copy) write what they should.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.api import kda_recover, step_from_inputs
from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, Workload, make_inputs
from tests.hostdata import bits, to_oracle
from tests.parity import STATE_ATOL, STATE_RTOL, to_device

pytestmark = pytest.mark.gpu


def verify_w(T=3, **kw):
    base = dict(name="rv", batch=21, heads=5, tokens=T, num_slots=21 * T + 30,
                conv_width=T + 2, slot_layout="verify", pad=3, seed=90 + T,
                gate_mode=1, has_bias=True)
    base.update(kw)
    return Workload(**base)


def run_step(inp, record):
    d = to_device(inp)
    d["record"] = int(record)
    B, H, T = d["batch"], d["heads"], d["tokens"]
    out = torch.empty((B * T, H * 128), dtype=torch.bfloat16, device="cuda")
    ru = rk = None
    if record:
        ru = torch.zeros((B, H, T, 128), dtype=torch.float32, device="cuda")
        rk = torch.zeros((B, H, T, 256), dtype=torch.bfloat16, device="cuda")
    step_from_inputs(d, out, rec_u=ru, rec_kg=rk)()
    torch.cuda.synchronize()
    return d, ru, rk, out


def free_slots(o, n):
    used = set(int(x) for x in np.asarray(o["slots"]).ravel())
    free = [s for s in range(1, o["num_slots"]) if s not in used]
    assert len(free) >= n
    return np.array(free[:n], np.int32)


def src_slots(o):
    B = o["batch"]
    return np.array([o["slots"][r, int(o["accepted"][r]) - 1] for r in range(B)], np.int32)


@pytest.mark.parametrize("T", [2, 4, 8])
def test_record_then_replay_equals_non_record_verify_bitwise(T):
    w = verify_w(T)
    inp = make_inputs(w)
    o = to_oracle(inp)
    d_plain, _, _, out_plain = run_step(inp, record=False)
    d_rec, ru, rk, out_rec = run_step(inp, record=True)
    # record mode computes the same outputs as the plain verify, bit for bit
    assert torch.equal(out_rec.view(torch.int16), out_plain.view(torch.int16))
    plain_state = d_plain["state"].cpu().numpy()
    src = src_slots(o)
    dst = free_slots(o, w.batch)
    rng = np.random.default_rng(T)
    acc = rng.integers(1, T + 1, size=w.batch).astype(np.int32)
    st = d_rec["state"]
    kda_recover(state=st, src_slots=torch.from_numpy(src).cuda(),
                dst_slots=torch.from_numpy(dst).cuda(),
                accepted=torch.from_numpy(acc).cuda(), rec_u=ru, rec_kg=rk,
                a_log=d_rec["a_log"], dt_bias=d_rec["dt_bias"],
                lower_bound=w.lower_bound)
    torch.cuda.synchronize()
    got = st.cpu().numpy()
    checked = 0
    for r in range(w.batch):
        if src[r] <= 0:
            assert np.array_equal(got[dst[r]], o["state"][dst[r]])  # padding
            continue
        want = plain_state[int(o["slots"][r, acc[r] - 1])]
        assert np.array_equal(got[dst[r]].view(np.uint32), want.view(np.uint32)), r
        checked += 1
    assert checked > 0


def test_replay_matches_oracle_on_gpu_records():
    T = 4
    w = verify_w(T, batch=17, heads=6, num_slots=17 * 4 + 40, seed=123)
    inp = make_inputs(w)
    o = to_oracle(inp)
    d_rec, ru, rk, _ = run_step(inp, record=True)
    src = src_slots(o)
    dst = free_slots(o, w.batch)
    acc = np.random.default_rng(7).integers(0, T + 1, size=w.batch).astype(np.int32)
    st = d_rec["state"]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_recover(state=st, src_slots=torch.from_numpy(src).cuda(),
                dst_slots=torch.from_numpy(dst).cuda(),
                accepted=torch.from_numpy(acc).cuda(), rec_u=ru, rec_kg=rk,
                a_log=d_rec["a_log"], dt_bias=d_rec["dt_bias"],
                lower_bound=w.lower_bound, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want, oerr = oracle.recover(state=o["state"], src_slots=src, dst_slots=dst,
                                accepted=acc, rec_u=ru.cpu().numpy(),
                                rec_kg=bits(rk), a_log=o["a_log"],
                                dt_bias=o["dt_bias"], lower_bound=o["lower_bound"])
    assert oerr == 0
    got = st.cpu().numpy()
    err_abs = np.abs(got.astype(np.float64) - want)
    assert np.all(err_abs <= STATE_ATOL + STATE_RTOL * np.abs(want))
    # pages nobody writes are untouched
    untouched = [s for s in range(w.num_slots) if s not in set(dst.tolist())]
    assert np.array_equal(got[untouched].view(np.uint32),
                          o["state"][untouched].view(np.uint32))


def test_replay_padding_errors_and_copy():
    T = 3
    w = verify_w(T, batch=6, heads=2, num_slots=60, pad=0, seed=5)
    inp = make_inputs(w)
    o = to_oracle(inp)
    d_rec, ru, rk, _ = run_step(inp, record=True)
    st = d_rec["state"]
    before = st.clone()
    src = np.array([0, 3, 99, 4, 5, 6], np.int32)
    dst = np.array([40, 41, 42, 43, 0, 45], np.int32)
    acc = np.array([1, 0, 1, 9, 1, 2], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_recover(state=st, src_slots=torch.from_numpy(src).cuda(),
                dst_slots=torch.from_numpy(dst).cuda(),
                accepted=torch.from_numpy(acc).cuda(), rec_u=ru, rec_kg=rk,
                a_log=d_rec["a_log"], dt_bias=d_rec["dt_bias"],
                lower_bound=w.lower_bound, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kl.KDA_DEVERR_SLOT | kl.KDA_DEVERR_ACCEPTED
    got, b = st.cpu(), before.cpu()
    assert torch.equal(got[40], b[40])          # src padding: nothing written
    assert torch.equal(got[41], b[3])           # accepted 0: copy of the checkpoint
    assert torch.equal(got[42], b[42])          # src beyond the pool: error, nothing
    assert torch.equal(got[43], b[43])          # accepted beyond T: error, nothing
    assert not torch.equal(got[45], b[45])      # a live replay wrote its page
    changed = [s for s in range(w.num_slots) if not torch.equal(got[s], b[s])]
    assert sorted(changed) == [41, 45]


def test_replay_full_size_record_workload_sampled():
    w = WORKLOADS["verify_q8_record_b64_h64"]
    inp = make_inputs(w)
    o = to_oracle(inp)
    d_rec, ru, rk, _ = run_step(inp, record=True)
    B, H, T = w.batch, w.heads, w.tokens
    # replay into a fresh pool region: grow the pool by B slots for the outputs
    st = torch.cat([d_rec["state"], torch.zeros((B, H, 128, 128), device="cuda")])
    src = src_slots(o)
    dst = np.arange(w.num_slots, w.num_slots + B, dtype=np.int32)
    acc = np.random.default_rng(11).integers(0, T + 1, size=B).astype(np.int32)
    kda_recover(state=st, src_slots=torch.from_numpy(src).cuda(),
                dst_slots=torch.from_numpy(dst).cuda(),
                accepted=torch.from_numpy(acc).cuda(), rec_u=ru, rec_kg=rk,
                a_log=d_rec["a_log"], dt_bias=d_rec["dt_bias"],
                lower_bound=w.lower_bound)
    torch.cuda.synchronize()
    got = st.cpu().numpy()
    sample = np.random.default_rng(3).choice(B, size=12, replace=False)
    pool = np.concatenate([o["state"], np.zeros((B, H, 128, 128), np.float32)])
    sub_src = np.where(np.isin(np.arange(B), sample), src, 0).astype(np.int32)
    want, _ = oracle.recover(state=pool, src_slots=sub_src, dst_slots=dst, accepted=acc,
                             rec_u=ru.cpu().numpy(), rec_kg=bits(rk),
                             a_log=o["a_log"], dt_bias=o["dt_bias"],
                             lower_bound=o["lower_bound"])
    for r in sample:
        if src[r] <= 0:
            continue
        g, t = got[dst[r]].astype(np.float64), want[dst[r]]
        assert np.all(np.abs(g - t) <= STATE_ATOL + STATE_RTOL * np.abs(t)), r


@pytest.mark.parametrize("full", [False, True])
def test_replay_shared_items_same_bits_as_fixed_ranges(full):
    """The replay with scheduler words (the items past the CTAs' ranges handed
    out one at a time) writes the same pages bit for bit as with contiguous
    ranges only, and leaves the words at zero; 96 requests x 8 heads (768
    items over at most one CTA per SM) and the full record workload."""
    w = (WORKLOADS["verify_q8_record_b64_h64"] if full else
         Workload(name="rs", batch=96, heads=8, tokens=6, num_slots=97, conv_width=8,
                  slot_layout="checkpoint", record=True, pad=9, seed=771))
    inp = make_inputs(w)
    o = to_oracle(inp)
    d_rec, ru, rk, _ = run_step(inp, record=True)
    B, H, T = w.batch, w.heads, w.tokens
    src = torch.from_numpy(src_slots(o)).cuda()
    dst = torch.arange(w.num_slots, w.num_slots + B, dtype=torch.int32, device="cuda")
    acc = torch.from_numpy(np.random.default_rng(12).integers(0, T + 1, size=B)
                           .astype(np.int32)).cuda()
    base = torch.cat([d_rec["state"], torch.zeros((B, H, 128, 128), device="cuda")])
    outs = []
    sched = torch.zeros(2, dtype=torch.int32, device="cuda")
    for kw in (dict(balance=False), dict(sched=sched), dict(sched=sched)):
        st = base.clone()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda_recover(state=st, src_slots=src, dst_slots=dst, accepted=acc, rec_u=ru,
                    rec_kg=rk, a_log=d_rec["a_log"], dt_bias=d_rec["dt_bias"],
                    lower_bound=w.lower_bound, err=err, **kw)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(st.view(torch.int32).cpu())
    assert sched.tolist() == [0, 0]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
