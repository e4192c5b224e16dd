"""Pools beyond 32-bit element offsets.

The same step runs twice: on a small pool (slots 1..n, parity-tested against
the oracle elsewhere) and on an 8.8 GB pool holding the same pages and conv
windows at its highest slots (page offsets past 2^31 elements).  Slot
numbering is only an address, so every result must be bit-identical: the
outputs, the records, the error word, and the pages and conv windows at the
relabelled slots.  Decode, verify and record steps on both kernel paths, and
the record replay and the access-pattern probe on the large pool.
"""
from __future__ import annotations

import pytest
import torch

from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.api import kda_recover, step_from_inputs
from linear_attention_recurrent_kda_gb300.probe import kda_probe_page_copy
from linear_attention_recurrent_kda_gb300.workloads import Workload, make_inputs
from tests.parity import to_device

pytestmark = pytest.mark.gpu

BIG = 4200     # slots of the large pool: 4200 x 32 heads x 64 KiB = 8.8 GB


def _run(d, path):
    B, H, T = d["batch"], d["heads"], d["tokens"]
    out = torch.full((B * T, H * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ru = rk = None
    if d["record"]:
        ru = torch.zeros((B, H, T, 128), dtype=torch.float32, device="cuda")
        rk = torch.zeros((B, H, T, 256), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step_from_inputs(d, out, rec_u=ru, rec_kg=rk, err=err, path=path)()
    torch.cuda.synchronize()
    return out, ru, rk, int(err.item())


def _enlarge(d):
    """The same inputs with pool slot s moved to BIG - n + s (n = pool size)."""
    n = d["num_slots"]
    shift = BIG - n
    e = dict(d)
    e["num_slots"] = BIG
    e["slots"] = torch.where(d["slots"] > 0, d["slots"] + shift, d["slots"])
    st = torch.empty((BIG,) + tuple(d["state"].shape[1:]), dtype=d["state"].dtype,
                     device="cuda")
    st[shift:].copy_(d["state"])
    cv = torch.empty((BIG,) + tuple(d["conv_state"].shape[1:]), dtype=d["conv_state"].dtype,
                     device="cuda")
    cv[shift:].copy_(d["conv_state"])
    e["state"], e["conv_state"] = st, cv
    return e, shift


CASES = {
    "decode": Workload("big_dec", batch=40, heads=32, tokens=1, num_slots=48, conv_width=3,
                       slot_layout="decode", pad=3, seed=501),
    "verify": Workload("big_ver", batch=12, heads=32, tokens=4, num_slots=12 * 4 + 5,
                       conv_width=6, slot_layout="verify", pad=1, seed=502),
    "record": Workload("big_rec", batch=10, heads=32, tokens=8, num_slots=12, conv_width=10,
                       slot_layout="checkpoint", pad=1, gate_mode=1, has_bias=True,
                       record=True, seed=503),
}


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("path", [kl.KDA_PATH_PERSISTENT, kl.KDA_PATH_SPLIT])
@pytest.mark.parametrize("case", sorted(CASES))
def test_relabelled_large_pool_gives_the_same_bits(case, path):
    inp = make_inputs(CASES[case])
    small = to_device(inp)
    big, shift = _enlarge(to_device(inp))
    assert big["state"].numel() > 2 ** 31
    a = _run(small, path)
    b = _run(big, path)
    for x, y in zip(a[:3], b[:3]):
        if x is not None:
            assert _same(x, y)
    assert a[3] == b[3]
    assert _same(small["state"], big["state"][shift:])
    assert _same(small["conv_state"], big["conv_state"][shift:])
    del big
    torch.cuda.empty_cache()


def test_replay_and_probe_on_large_pool():
    w = CASES["record"]
    inp = make_inputs(w)
    small = to_device(inp)
    big, shift = _enlarge(to_device(inp))
    _, ru, rk, _ = _run(small, kl.KDA_PATH_PERSISTENT)
    B, T = w.batch, w.tokens
    src = torch.tensor([int(inp["slots"][r, int(inp["accepted"][r]) - 1]) for r in range(B)],
                       dtype=torch.int32, device="cuda")
    acc = torch.arange(B, dtype=torch.int32, device="cuda") % (T + 1)
    for pool, off in ((small, 0), (big, shift)):
        s = torch.where(src > 0, src + off, src)
        kda_recover(state=pool["state"], src_slots=s, dst_slots=s, accepted=acc, rec_u=ru,
                    rec_kg=rk, a_log=pool["a_log"], dt_bias=pool["dt_bias"],
                    lower_bound=w.lower_bound)
    torch.cuda.synchronize()
    assert _same(small["state"], big["state"][shift:])
    before = big["state"][shift:].clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda_probe_page_copy(state=big["state"], slots=torch.where(src > 0, src + shift, src),
                        err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _same(before, big["state"][shift:])
    del big
    torch.cuda.empty_cache()
