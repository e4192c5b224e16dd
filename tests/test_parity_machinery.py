"""The GPU-vs-oracle comparison (tests/parity.py) checked on the CPU.

The oracle's float64 mode is a second correct implementation of the step (it
rounds at the same BF16 points but computes everything else in double), so
`compare` must accept its results in place of the GPU's; results with a
planted deviation must be rejected."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from linear_attention_recurrent_kda_gb300.workloads import Workload, make_inputs
from tests import hostdata
from tests.hostdata import to_oracle
from tests.parity import compare, same_bits, silu_band, unanchored


def fake_gpu(inp):
    o = to_oracle(inp)
    r = oracle.run(o, mode="f64", want_intermediates=True)
    res = {"output": r["output"], "state": r["state"], "conv_state": r["conv_state"],
           "err": r["err"], "dbg": r["inter"]}
    if o["record"]:
        res["rec_u"], res["rec_kg"] = r["rec_u"], r["rec_kg"]
    return res


def wl(**kw):
    base = dict(name="m", batch=6, heads=3, tokens=1, num_slots=16, conv_width=3,
                slot_layout="decode", pad=1, seed=77)
    base.update(kw)
    return Workload(**base)


@pytest.mark.parametrize("w", [wl(), wl(tokens=3, slot_layout="verify", conv_width=5,
                                        num_slots=20, gate_mode=1, has_bias=True),
                               wl(tokens=4, slot_layout="checkpoint", conv_width=6,
                                  record=True)])
def test_second_implementation_passes(w):
    inp = make_inputs(w)
    compare(inp, fake_gpu(inp))
    items = np.array([0, 4, 7, 11, 17])
    compare(inp, fake_gpu(inp), items=items)


@pytest.mark.parametrize("plant", ["state", "output", "conv", "dbg", "pad", "err"])
def test_planted_deviation_fails(plant):
    w = wl(tokens=2, slot_layout="verify", conv_width=4, num_slots=20)
    inp = make_inputs(w)
    g = fake_gpu(inp)
    o = to_oracle(inp)
    r = 0 if o["slots"][0, int(o["accepted"][0]) - 1] > 0 else 1
    if plant == "state":
        s = int(o["slots"][r, 0])
        g["state"][s, 0, 3, 5] += 1e-3
    elif plant == "output":
        g["output"][r * 2, 7] ^= 0x0004       # a few ulps
    elif plant == "conv":
        s = int(o["slots"][r, 0])
        g["conv_state"][s, 0, 1] ^= 0x0001
    elif plant == "dbg":
        g["dbg"][r, 0, 0, 1, 3] ^= 0x0002
    elif plant == "pad":
        pr = [q for q in range(w.batch) if o["slots"][q, int(o["accepted"][q]) - 1] <= 0][0]
        g["output"][pr * 2, 0] = 0x3F80
    elif plant == "err":
        g["err"] = 1
    with pytest.raises(AssertionError):
        compare(inp, g)


def test_reports_carry_the_unanchored_numbers():
    w = wl(tokens=3, slot_layout="verify", conv_width=5, num_slots=20)
    inp = make_inputs(w)
    st = compare(inp, fake_gpu(inp))
    for key in ("unanchored_out_max_ulp", "unanchored_state_worst_frac_of_tol",
                "unanchored_state_beyond_tol", "unanchored_flips"):
        assert key in st
    # without a dbg dump (a launch as a caller makes it) the report still works
    g = fake_gpu(inp)
    del g["dbg"]
    rep = unanchored(inp, g)
    assert rep["unanchored_out_max_ulp"] >= 0 and "unanchored_flips" not in rep


def test_same_bits_catches_any_difference():
    inp = make_inputs(wl())
    a, b = fake_gpu(inp), fake_gpu(inp)
    same_bits(a, b)
    b["state"] = b["state"].copy()
    b["state"].reshape(-1)[123] = np.nextafter(b["state"].reshape(-1)[123], np.float32(9))
    with pytest.raises(AssertionError):
        same_bits(a, b)


def test_one_ulp_flip_away_from_a_midpoint_fails():
    """A one-ulp difference of a BF16 q where the oracle's unrounded value is
    far from the midpoint is not a rounding difference: rejected."""
    w = wl(pad=0)
    inp = make_inputs(w)
    g = fake_gpu(inp)
    o = to_oracle(inp)
    r = oracle.run(o, mode="f32", want_intermediates=True)
    pre = r["pre"][..., 0, :]                       # q before rounding
    val = hostdata.bf16_bits_to_f64(r["inter"][..., 0, :])
    rel = np.abs(pre - val) / np.maximum(np.abs(val), 1e-30)
    idx = np.unravel_index(np.argmin(rel + (np.abs(val) < 1e-3)), rel.shape)
    g["dbg"][idx[0], idx[1], idx[2], 0, idx[3]] ^= 0x0001
    with pytest.raises(AssertionError, match="SiLU flip outside band"):
        compare(inp, g)


@pytest.mark.parametrize("sign_e", [-1, 1])
@pytest.mark.parametrize("sign_d", [-1, 1])
def test_silu_band_covers_the_instruction_error_bounds(sign_e, sign_d):
    """Worst-case kernel SiLU (exp2 and divide at the edges of their error
    bounds, argument and constant rounded to FP32) against the oracle's
    (double exp rounded once, FP32 add and divide): the difference stays
    within silu_band for arguments across the whole range the step meets."""
    a = np.concatenate([np.linspace(-100, 100, 20001), -np.logspace(-6, 2, 500),
                        np.logspace(-6, 2, 500)]).astype(np.float32)
    a64 = a.astype(np.float64)
    # oracle (f32 mode)
    with np.errstate(over="ignore"):
        e_o = np.exp(-a64).astype(np.float32)
        den_o = (np.float32(1) + e_o).astype(np.float32)
        y_o = (a / den_o).astype(np.float32).astype(np.float64)
    # kernel: t1 = fl(-a * fl(log2 e)); e = 2^t1 (1 +- 2^-22); den = fl(1 + e);
    # y = (a / den)(1 +- 2^-22)
    l2e = np.float32(1.4426950408889634)
    t1 = (-a * l2e).astype(np.float32).astype(np.float64)
    with np.errstate(over="ignore"):
        e_g = (np.exp2(t1) * (1 + sign_e * 2.0 ** -22)).astype(np.float32)
        den_g = (np.float32(1) + e_g).astype(np.float32).astype(np.float64)
        y_g = a64 / den_g * (1 + sign_d * 2.0 ** -22)
    ok = np.isfinite(y_o) & (np.abs(y_o) > 0)
    diff = np.abs(y_g[ok] - y_o[ok])
    assert np.all(diff <= silu_band(a64[ok]) * np.abs(y_o[ok]))
    # and the band is tight for moderate arguments: a few FP32 ulps
    assert silu_band(np.array([3.0]))[0] < 16 * 2.0 ** -24
