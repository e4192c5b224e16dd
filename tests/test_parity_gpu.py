"""GPU parity of the KDA decode/verify library against the CPU oracle.

Every test runs the CUDA path through the C ABI (``libkda_gb300.so`` via the
ctypes binding) on seeded synthetic inputs and compares it with the oracle
element by element, using the anchored comparison of tests/parity.py.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, Workload, make_inputs
from tests.hostdata import bits, to_oracle
from tests.parity import compare, run_gpu, same_bits, to_device, unanchored

pytestmark = pytest.mark.gpu


def small(**kw) -> Workload:
    base = dict(name="small", batch=37, heads=9, tokens=1, num_slots=64,
                conv_width=3, slot_layout="decode", pad=5, seed=21)
    base.update(kw)
    return Workload(**base)


def check(w: Workload, mutate=None, items=None):
    inp = make_inputs(w)
    if mutate:
        mutate(inp)
    gpu = run_gpu(inp)
    return compare(inp, gpu, items=items)


# ---------------------------------------------------------------- decode

def test_decode_b4_h8_full():
    check(WORKLOADS["decode_b4_h8"])


def test_decode_b64_h32_pad8_full():
    check(WORKLOADS["decode_b64_h32_pad8"])


def test_decode_ragged_tail_many_items_per_cta():
    # 333 items over <= 152 CTAs: 2-3 items each, uneven split, padding mixed in
    check(small())


def test_decode_many_items_per_cta_crosses_heads():
    check(small(batch=200, heads=5, num_slots=256, pad=17, seed=22))


@pytest.mark.parametrize("tokens", [1, 3])
def test_mostly_padding_balanced_ranges(tokens):
    """Two thirds of the requests padded, live ones bunched at the end: each
    CTA's range holds the same number of live items, padding rides along."""
    lay = dict(slot_layout="decode") if tokens == 1 else dict(
        slot_layout="verify", conv_width=tokens + 2)
    w = small(tokens=tokens, batch=300, heads=4, num_slots=300 * tokens + 2, pad=200,
              seed=280 + tokens, **lay)

    def mutate(inp):
        live = inp["slots"].reshape(300, -1)[:, 0] > 0 if tokens > 1 else inp["slots"] > 0
        order = torch.argsort(live.to(torch.int8), stable=True)   # padding first
        inp["slots"] = inp["slots"][order].contiguous()
        if tokens > 1:
            inp["accepted"] = inp["accepted"][order].contiguous()

    check(w, mutate)


def test_batch_beyond_the_balanced_scan():
    """More requests than every CTA scans at start: equal item counts."""
    check(small(batch=8200, heads=1, num_slots=8201, pad=8000, seed=290))


def test_decode_all_padding():
    w = small(batch=6, heads=4, pad=6)
    st = check(w)
    assert st["out_max_ulp"] == 0


def test_decode_zero_beta_zero_lower_bound_keeps_state_bits():
    w = small(batch=20, heads=3, pad=0, lower_bound=0.0)

    def mutate(inp):
        inp["beta"] = torch.full_like(inp["beta"], float("-inf"))

    inp = make_inputs(w)
    mutate(inp)
    gpu = run_gpu(inp)
    compare(inp, gpu)
    o = to_oracle(inp)
    for r in range(w.batch):
        s = int(o["slots"][r])
        assert np.array_equal(gpu["state"][s].view(np.uint32), o["state"][s].view(np.uint32))


def test_decode_repeat_is_deterministic():
    w = small(batch=50, heads=4)
    inp = make_inputs(w)
    a = run_gpu(inp)
    b = run_gpu(inp)
    for k in ("output", "state", "conv_state", "dbg"):
        assert np.array_equal(a[k], b[k]), k


def test_decode_two_steps_chain():
    """Two consecutive decode calls on the same pools match two oracle steps."""
    w = small(batch=16, heads=4, pad=2)
    inp = make_inputs(w)
    d = to_device(inp)
    from linear_attention_recurrent_kda_gb300.api import step_from_inputs
    B, H = w.batch, w.heads
    out = torch.empty((B, H * 128), dtype=torch.bfloat16, device="cuda")
    dbg = torch.zeros((B, H, 1, 4, 128), dtype=torch.bfloat16, device="cuda")
    step = step_from_inputs(d, out, dbg=dbg)
    step()
    torch.cuda.synchronize()
    mid = dict(inp)
    mid["state"] = d["state"].cpu().clone()
    mid["conv_state"] = d["conv_state"].cpu().clone()
    step()
    torch.cuda.synchronize()
    gpu = {"output": bits(out), "state": d["state"].cpu().numpy(),
           "conv_state": bits(d["conv_state"]), "err": 0, "dbg": bits(dbg)}
    compare(mid, gpu)


# ---------------------------------------------------------------- verify

@pytest.mark.parametrize("tokens", [2, 3, 4, 5, 8])
def test_verify_per_token_writes(tokens):
    w = small(tokens=tokens, slot_layout="verify", conv_width=tokens + 2,
              batch=23, heads=7, num_slots=23 * tokens + 5, pad=3, seed=30 + tokens)
    check(w)


def test_verify_accepted_extremes_and_skipped_targets():
    T = 4
    w = small(tokens=T, slot_layout="verify", conv_width=T + 3, batch=12, heads=6,
              num_slots=12 * T + 1, pad=0, seed=40)

    def mutate(inp):
        acc = inp["accepted"]
        acc[:6] = 1
        acc[6:] = T
        sl = inp["slots"]
        sl[0, 2] = 0        # token 2 of request 0 not written
        sl[7, 1] = -3       # token 1 of request 7 not written

    check(w, mutate)


@pytest.mark.parametrize("tokens,gate_mode,has_bias", [(2, 0, False), (4, 1, True),
                                                        (8, 1, True), (8, 0, False)])
def test_record_mode(tokens, gate_mode, has_bias):
    w = small(tokens=tokens, slot_layout="checkpoint", conv_width=tokens + 2,
              record=True, gate_mode=gate_mode, has_bias=has_bias, batch=19,
              heads=6, num_slots=25, pad=2, seed=50 + tokens)
    check(w)


@pytest.mark.parametrize("record", [False, True])
@pytest.mark.parametrize("tokens", [2, 3, 4, 5, 6, 7, 8])
def test_every_token_count_with_a_wide_window(tokens, record):
    """Every verify instantiation (T = 2..8, with and without records), the
    conv window wider than T + 2 (the extra columns keep their values)."""
    extra = 1 + tokens % 3
    if record:
        w = small(tokens=tokens, slot_layout="checkpoint", conv_width=tokens + 2 + extra,
                  record=True, gate_mode=tokens % 2, has_bias=tokens % 3 == 0, batch=11,
                  heads=5, num_slots=14, pad=1, seed=200 + tokens)
    else:
        w = small(tokens=tokens, slot_layout="verify", conv_width=tokens + 2 + extra,
                  gate_mode=tokens % 2, has_bias=tokens % 3 == 1, batch=11, heads=5,
                  num_slots=11 * tokens + 2, pad=1, seed=220 + tokens)
    check(w)


@pytest.mark.parametrize("case", ["x_saturated", "x_zero", "state_large", "beta_saturated"])
@pytest.mark.parametrize("tokens", [1, 4])
def test_extreme_inputs(case, tokens):
    """Inputs at the edges of the functions' ranges: SiLU saturated (x * 20),
    all-zero x (q = k = 0: the L2 norms fall back on their 1e-6), state pages
    scaled by 100, beta logits of +-20 (sigmoid saturated)."""
    if tokens == 1:
        w = small(batch=13, heads=4, num_slots=20, pad=1, seed=260)
    else:
        w = small(tokens=4, slot_layout="verify", conv_width=6, batch=9, heads=3,
                  num_slots=9 * 4 + 2, pad=1, seed=261)

    def mutate(inp):
        if case == "x_saturated":
            inp["x"] = (inp["x"].float() * 20.0).to(torch.bfloat16)
        elif case == "x_zero":
            inp["x"] = torch.zeros_like(inp["x"])
            inp["conv_state"] = torch.zeros_like(inp["conv_state"])
            if inp.get("conv_bias") is not None:
                inp["conv_bias"] = torch.zeros_like(inp["conv_bias"])
        elif case == "state_large":
            inp["state"] = inp["state"] * 100.0
        else:
            sign = torch.where(torch.arange(inp["beta"].numel()) % 2 == 0, 1.0, -1.0)
            inp["beta"] = (sign.view_as(inp["beta"]) * 20.0).to(torch.bfloat16)

    check(w, mutate)


def test_many_heads_decode():
    check(small(batch=3, heads=96, num_slots=8, pad=0, seed=240))


def test_gate_mode_1_and_bias_decode():
    check(small(gate_mode=1, has_bias=True, seed=60))


def test_error_items_flag_and_pad():
    T = 3
    w = small(tokens=T, slot_layout="verify", conv_width=T + 2, batch=8, heads=4,
              num_slots=8 * T + 1, pad=0, seed=70)

    def mutate(inp):
        inp["slots"][1, 1] = 10_000          # target beyond the pool
        inp["accepted"][2] = 0                # accepted out of range
        inp["accepted"][3] = T + 1
        inp["slots"][4, 0] = -1               # live item whose conv slot is invalid
        inp["accepted"][4] = 2

    inp = make_inputs(w)
    mutate(inp)
    gpu = run_gpu(inp)
    assert gpu["err"] == kl.KDA_DEVERR_SLOT | kl.KDA_DEVERR_ACCEPTED
    compare(inp, gpu)


# --------------------------------------------------- the five named workloads

@pytest.mark.parametrize("path", [kl.KDA_PATH_AUTO, kl.KDA_PATH_SPLIT])
@pytest.mark.parametrize("name", ["decode_b256_h32", "verify_q4_b128_h32",
                                  "verify_q8_record_b64_h64"])
def test_full_size_workloads_sampled(name, path):
    """Full-size launch as a caller makes it (no dbg buffer; the automatic
    path is the one the benchmark times): its pools, outputs, records and
    error word equal, bit for bit, those of a launch with the dbg buffer on
    the same inputs, which the anchored comparison checks against the oracle
    on a seeded sample of 1024 items one by one (plus every padded item); the
    product launch itself is also compared with the oracle unanchored."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    rng = np.random.default_rng(5)
    items = np.sort(rng.choice(w.items, size=1024, replace=False))
    prod = run_gpu(inp, dbg=False, path=path)
    rep = unanchored(inp, prod, items=items)
    checked = run_gpu(inp, dbg=True, path=path)
    same_bits(prod, checked)
    del prod
    st = compare(inp, checked, items=items)
    print(name, path, st, rep)


PRODUCT_CASES = {
    "decode_pad": dict(batch=37, heads=9, pad=5, seed=21),
    "decode_gm1_bias": dict(batch=40, heads=6, gate_mode=1, has_bias=True, seed=60),
    "verify4_skips": dict(tokens=4, slot_layout="verify", conv_width=7, batch=23,
                          heads=7, num_slots=23 * 4 + 5, pad=3, seed=34),
    "record8_gm1_bias": dict(tokens=8, slot_layout="checkpoint", conv_width=10,
                             record=True, gate_mode=1, has_bias=True, batch=19,
                             heads=6, num_slots=25, pad=2, seed=58),
}


@pytest.mark.parametrize("path", [kl.KDA_PATH_PERSISTENT, kl.KDA_PATH_SPLIT])
@pytest.mark.parametrize("case", list(PRODUCT_CASES))
def test_launch_without_dbg_is_the_checked_launch(case, path):
    """Every item compared: a launch without the dbg buffer gives the bits of
    the dbg launch, which passes the anchored comparison."""
    w = small(**PRODUCT_CASES[case])
    inp = make_inputs(w)
    prod = run_gpu(inp, dbg=False, path=path)
    checked = run_gpu(inp, dbg=True, path=path)
    same_bits(prod, checked)
    st = compare(inp, checked)
    print(case, path, st)


# ------------------------------------------------------------ host errors

def _base_args(d, out):
    from linear_attention_recurrent_kda_gb300.api import step_from_inputs
    return step_from_inputs(d, out).args


def test_host_side_errors_launch_nothing():
    w = small(batch=4, heads=2, pad=0)
    inp = make_inputs(w)
    d = to_device(inp)
    out = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    before = d["state"].clone()

    def code(mod, entry="kda_decode"):
        a = _base_args(d, out)
        mod(a)
        return kl.call(entry, a, 0)

    assert code(lambda a: setattr(a, "tokens", 0)) == kl.KDA_ERR_TOKENS
    assert code(lambda a: setattr(a, "tokens", 9), "kda_verify") == kl.KDA_ERR_TOKENS
    assert code(lambda a: setattr(a, "tokens", 2)) == kl.KDA_ERR_TOKENS
    assert code(lambda a: None, "kda_verify") == kl.KDA_ERR_TOKENS
    assert code(lambda a: setattr(a, "gate_mode", 2)) == kl.KDA_ERR_GATE_MODE
    assert code(lambda a: setattr(a, "state", None)) == kl.KDA_ERR_NULL_POINTER
    assert code(lambda a: setattr(a, "conv_width", 2)) == kl.KDA_ERR_CONV_WIDTH
    assert code(lambda a: setattr(a, "conv_width", 4000)) == kl.KDA_ERR_CONV_WIDTH
    assert code(lambda a: setattr(a, "state", a.state + 4)) == kl.KDA_ERR_ALIGNMENT
    assert code(lambda a: setattr(a, "num_slots", 0)) == kl.KDA_ERR_SHAPE
    assert code(lambda a: setattr(a, "batch", 0)) == kl.KDA_SUCCESS   # no-op
    torch.cuda.synchronize()
    assert torch.equal(before, d["state"])
    assert not out.any()


def test_record_needs_tokens():
    w = small(batch=2, heads=2, pad=0)
    d = to_device(make_inputs(w))
    out = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    a = _base_args(d, out)
    a.record = 1
    assert kl.call("kda_decode", a, 0) == kl.KDA_ERR_RECORD


def test_nondefault_stream():
    w = small(batch=30, heads=4)
    inp = make_inputs(w)
    s = torch.cuda.Stream()
    gpu = run_gpu(inp, stream=s)
    compare(inp, gpu)
