"""Pins of the CPU oracle against things other than itself.

The oracle (oracle/kda_oracle.c) restates the KDA decode/verify step of the
vLLM API page "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide"
(KdaWide).  These tests hold it to closed forms, invariants, library routines
and a float64 matrix-form brute force (tests/textbook.py), chosen so that a
dropped term, a wrong sign, a wrong index or a transposed operand anywhere in
it fails at least one of them.  CPU only.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrent_kda_gb300.workloads import Workload, make_inputs
from tests import textbook as tb
from tests.hostdata import (bf16_bits_to_f64, bf16_ulp_diff, f32_to_bf16_bits,
                            to_oracle)

F32_EPS = 2.0 ** -24


def tiny(**kw) -> Workload:
    base = dict(name="tiny", batch=3, heads=2, tokens=1, num_slots=8,
                conv_width=3, slot_layout="decode", dk=8, rank=16, seed=7)
    base.update(kw)
    return Workload(**base)


def prepare(w: Workload, mutate=None):
    inp = make_inputs(w)
    if mutate is not None:
        mutate(inp)
    return inp, to_oracle(inp)


def resolve(o, r):
    """(state slot, conv slot, window offset) of request r, or None (pad)."""
    T = o["tokens"]
    if T == 1:
        s = int(o["slots"][r])
        return (s, s, 0) if s > 0 else None
    a = int(o["accepted"][r])
    s = int(o["slots"][r, a - 1])
    return (s, int(o["slots"][r, 0]), a - 1) if s > 0 else None


def f64(bits):
    return bf16_bits_to_f64(bits)


# ---------------------------------------------------------------- rounding

@pytest.mark.parametrize("gate_mode", [0, 1])
def test_bf16_rounding_f32_mode_matches_torch(gate_mode):
    w = tiny(dk=16, rank=32, gate_mode=gate_mode, batch=4, heads=3)
    _, o = prepare(w)
    res = oracle.run(o, mode="f32", want_intermediates=True)
    pre = res["pre"].astype(np.float32)          # exact: f32-mode values
    assert np.array_equal(res["pre"], pre.astype(np.float64))
    assert np.array_equal(res["inter"], f32_to_bf16_bits(pre))


def test_bf16_rounding_f64_mode_nearest_even():
    w = tiny(dk=8, rank=16, batch=2, heads=2)
    _, o = prepare(w)
    res = oracle.run(o, mode="f64", want_intermediates=True)
    assert np.array_equal(res["inter"].ravel(), tb.rne_bf16_bits(res["pre"]))


# --------------------------------------------------------- conv + SiLU (a3)

def _conv_reference(o, r, h, part, c, off, T, bias):
    D, H = o["dk"], o["heads"]
    dim = H * D
    ch = part * dim + h * D + c
    cs = resolve(o, r)[1]
    taps = f64(o["conv_state"][cs, ch, off:off + 3])
    xs = f64(o["x"][r * T:(r + 1) * T, ch])
    wt = f64(o["conv_weight"][part, :, h * D + c])
    b = f64(o["conv_bias"][ch]) if bias else 0.0
    return tb.causal_conv4(taps, xs, wt, b)


@pytest.mark.parametrize("tokens,has_bias", [(1, False), (3, True), (5, False)])
def test_conv_silu_against_sliding_window(tokens, has_bias):
    lay = "decode" if tokens == 1 else "verify"
    w = tiny(tokens=tokens, slot_layout=lay, has_bias=has_bias,
             conv_width=tokens + 2, num_slots=3 * tokens + 1 if tokens > 1 else 8)
    _, o = prepare(w)
    r64 = oracle.run(o, mode="f64", want_intermediates=True)
    r32 = oracle.run(o, mode="f32", want_intermediates=True)
    for r in range(w.batch):
        res = resolve(o, r)
        if res is None:
            continue
        off = res[2]
        for h in range(w.heads):
            for part in range(3):
                for c in range(w.dk):
                    a = _conv_reference(o, r, h, part, c, off, tokens, has_bias)
                    y = tb.silu(a)
                    got64 = r64["pre"][r, h, :, part, c]
                    got32 = r32["pre"][r, h, :, part, c]
                    np.testing.assert_allclose(got64, y, rtol=1e-13, atol=1e-15)
                    np.testing.assert_allclose(got32, y, rtol=8 * F32_EPS,
                                               atol=1e-30)
                    # the SiLU argument the oracle reports is the conv sum
                    np.testing.assert_allclose(r64["silu_in"][r, h, :, part, c], a,
                                               rtol=1e-13, atol=1e-15)
                    np.testing.assert_allclose(r32["silu_in"][r, h, :, part, c], a,
                                               rtol=8 * F32_EPS, atol=1e-6)


@pytest.mark.parametrize("tap", [0, 1, 2, 3])
def test_conv_one_hot_tap_selects_window_element(tap):
    T = 3
    w = tiny(tokens=T, slot_layout="verify", conv_width=T + 2, num_slots=10)

    def one_hot(inp):
        cw = torch.zeros_like(inp["conv_weight"], dtype=torch.float32)
        cw[:, tap, :] = 1.0
        inp["conv_weight"] = cw.to(torch.bfloat16)

    _, o = prepare(w, one_hot)
    res = oracle.run(o, mode="f64", want_intermediates=True)
    D, H = w.dk, w.heads
    for r in range(w.batch):
        s, cs, off = resolve(o, r)
        for h in range(H):
            for part in range(3):
                ch = part * H * D + h * D + np.arange(D)
                win = np.concatenate(
                    [f64(o["conv_state"][cs][ch, off:off + 3]).T,
                     f64(o["x"][r * T:(r + 1) * T][:, ch])], axis=0)
                for t in range(T):
                    np.testing.assert_allclose(
                        res["pre"][r, h, t, part], tb.silu(win[t + tap]),
                        rtol=1e-13, atol=1e-300)
    # silu(0) = 0 exactly
    assert tb.silu(0.0) == 0.0


# ------------------------------------------------------------ gate (a4)

@pytest.mark.parametrize("gate_mode", [0, 1])
def test_gate_projection_within_summation_bound(gate_mode):
    w = tiny(dk=16, rank=32, tokens=2, slot_layout="verify", conv_width=4,
             num_slots=7, gate_mode=gate_mode)
    _, o = prepare(w)
    r32 = oracle.run(o, mode="f32", want_intermediates=True)
    r64 = oracle.run(o, mode="f64", want_intermediates=True)
    fb = f64(o["f_b"])
    fa = f64(o["f_a"])
    exact = fa @ fb.T                       # [B*T, dim]
    mag = np.abs(fa) @ np.abs(fb).T
    R, T, D = w.rank, w.tokens, w.dk
    for r in range(w.batch):
        if resolve(o, r) is None:
            continue
        for h in range(w.heads):
            for t in range(T):
                e = exact[r * T + t, h * D:(h + 1) * D]
                m = mag[r * T + t, h * D:(h + 1) * D]
                g32 = r32["pre"][r, h, t, 3]
                g64 = r64["pre"][r, h, t, 3]
                assert np.all(np.abs(g32 - e) <= R * F32_EPS * m + 1e-30)
                assert np.all(np.abs(g64 - e) <= 1e-13 * m + 1e-300)


def test_gate_one_hot_rows_copy_f_a():
    w = tiny(dk=8, rank=16)

    def one_hot(inp):
        fb = torch.zeros(w.heads * w.dk, w.rank)
        for f in range(w.heads * w.dk):
            fb[f, (3 * f + 1) % w.rank] = 1.0
        inp["f_b"] = fb.to(torch.bfloat16)

    _, o = prepare(w, one_hot)
    res = oracle.run(o, mode="f32", want_intermediates=True)
    for r in range(w.batch):
        if resolve(o, r) is None:
            continue
        for h in range(w.heads):
            for f in range(w.dk):
                col = (3 * (h * w.dk + f) + 1) % w.rank
                assert res["inter"][r, h, 0, 3, f] == o["f_a"][r, col]


def test_gate_modes_agree_up_to_rounding():
    w = tiny(dk=16, rank=32)
    _, o = prepare(w)
    a = oracle.run(o, mode="f32", want_intermediates=True)
    b = oracle.run(dict(o, gate_mode=1), mode="f32", want_intermediates=True)
    fb, fa = f64(o["f_b"]), f64(o["f_a"])
    mag = np.abs(fa) @ np.abs(fb).T
    for r in range(w.batch):
        for h in range(w.heads):
            m = mag[r, h * w.dk:(h + 1) * w.dk]
            d = np.abs(a["pre"][r, h, 0, 3] - b["pre"][r, h, 0, 3])
            assert np.all(d <= 2 * w.rank * F32_EPS * m)


# --------------------------------- decay, beta, norms, recurrence (a4-a8)

def _item_textbook(o, inter, r, h, T, record=False):
    """Float64 matrix-form replay of one item from the oracle's BF16
    intermediates.  Returns per-token states (as [i][j] pages), o, u."""
    D, H = o["dk"], o["heads"]
    s = resolve(o, r)[0]
    S = o["state"][s, h].astype(np.float64).T        # [j][i]
    pages, outs, us = [], [], []
    for t in range(T):
        q = f64(inter[r, h, t, 0])
        k = f64(inter[r, h, t, 1])
        v = f64(inter[r, h, t, 2])
        g = f64(inter[r, h, t, 3])
        d = tb.decay(float(o["a_log"][h]), g,
                     o["dt_bias"][h * D:(h + 1) * D].astype(np.float64),
                     float(o["lower_bound"]))
        beta = tb.sigmoid(f64(o["beta"][r * T + t, h]))
        qh = tb.l2_normalise(q, scale=float(np.float32(o["scale"])))
        kh = tb.l2_normalise(k)
        S, u = tb.delta_rule(S, d, kh, v, beta)
        pages.append(S.T.copy())
        outs.append(S.T @ qh)
        us.append(u)
    return pages, outs, us


@pytest.mark.parametrize("dk,tokens", [(4, 1), (8, 1), (8, 3), (4, 2)])
def test_recurrence_matches_matrix_form_delta_rule(dk, tokens):
    lay = "decode" if tokens == 1 else "verify"
    w = tiny(dk=dk, rank=2 * dk, tokens=tokens, slot_layout=lay,
             conv_width=tokens + 2, num_slots=3 * tokens + 2, heads=2)
    _, o = prepare(w)
    res = oracle.run(o, mode="f64", want_intermediates=True)
    for r in range(w.batch):
        if resolve(o, r) is None:
            continue
        for h in range(w.heads):
            pages, outs, _ = _item_textbook(o, res["inter"], r, h, tokens)
            for t in range(tokens):
                np.testing.assert_allclose(res["o"][r, h, t], outs[t],
                                           rtol=1e-11, atol=1e-13)
                tgt = int(o["slots"][r]) if tokens == 1 else int(o["slots"][r, t])
                if tokens == 1 or tgt > 0:
                    if tokens > 1 and t < tokens - 1 and any(
                            int(o["slots"][r, u]) == tgt for u in range(t + 1, tokens)):
                        continue
                    np.testing.assert_allclose(
                        res["state"][tgt, h], pages[t].astype(np.float32),
                        rtol=2 * F32_EPS, atol=1e-30)


def test_record_mode_u_and_records():
    T = 3
    w = tiny(dk=8, rank=16, tokens=T, slot_layout="checkpoint", conv_width=T + 2,
             num_slots=5, record=True, gate_mode=1, has_bias=True, pad=1)
    _, o = prepare(w)
    state0 = o["state"].copy()
    res = oracle.run(o, mode="f64", want_intermediates=True)
    assert np.array_equal(res["state"], state0)      # record never writes state
    for r in range(w.batch):
        if resolve(o, r) is None:
            assert not res["rec_kg"][r].any() and not res["rec_u"][r].any()
            continue
        for h in range(w.heads):
            _, _, us = _item_textbook(o, res["inter"], r, h, T, record=True)
            for t in range(T):
                np.testing.assert_allclose(res["rec_u"][r, h, t],
                                           np.float32(us[t]), rtol=4 * F32_EPS,
                                           atol=1e-12)
                assert np.array_equal(res["rec_kg"][r, h, t, :w.dk],
                                      res["inter"][r, h, t, 1])
                assert np.array_equal(res["rec_kg"][r, h, t, w.dk:],
                                      res["inter"][r, h, t, 3])


def _neg_inf_beta(inp):
    inp["beta"] = torch.full_like(inp["beta"], float("-inf"))


def test_zero_beta_zero_lower_bound_leaves_state_bit_identical():
    for tokens in (1, 3):
        lay = "decode" if tokens == 1 else "verify"
        w = tiny(dk=16, rank=16, tokens=tokens, slot_layout=lay,
                 conv_width=tokens + 2, num_slots=3 * tokens + 2,
                 lower_bound=0.0)
        _, o = prepare(w, _neg_inf_beta)
        for mode in ("f32", "f64"):
            res = oracle.run(o, mode=mode, want_intermediates=True)
            for r in range(w.batch):
                sel = resolve(o, r)
                if sel is None:
                    continue
                for h in range(w.heads):
                    page = o["state"][sel[0], h]
                    tg = ([sel[0]] if tokens == 1 else
                          [int(x) for x in o["slots"][r] if x > 0])
                    for tgt in tg:
                        assert np.array_equal(res["state"][tgt, h], page)
                    # o = S^T q_hat with the unchanged state
                    q = f64(res["inter"][r, h, 0, 0])
                    qh = tb.l2_normalise(q, scale=float(np.float32(o["scale"])))
                    np.testing.assert_allclose(
                        res["o"][r, h, 0], page.astype(np.float64) @ qh,
                        rtol=1e-5 if mode == "f32" else 1e-11, atol=1e-6)


def test_zero_gate_input_decays_by_exp_half_lower_bound():
    T = 3
    w = tiny(dk=8, rank=16, tokens=T, slot_layout="verify", conv_width=T + 2,
             num_slots=11, lower_bound=-3.0)

    def mutate(inp):
        _neg_inf_beta(inp)
        inp["f_a"] = torch.zeros_like(inp["f_a"])
        inp["dt_bias"] = torch.zeros_like(inp["dt_bias"])

    _, o = prepare(w, mutate)
    res = oracle.run(o, mode="f64")
    for r in range(w.batch):
        sel = resolve(o, r)
        if sel is None:
            continue
        for h in range(w.heads):
            page = o["state"][sel[0], h].astype(np.float64)
            for t in range(T):
                tgt = int(o["slots"][r, t])
                want = page * np.exp(-1.5) ** (t + 1)
                np.testing.assert_allclose(res["state"][tgt, h], want,
                                           rtol=2 * F32_EPS, atol=1e-30)


def test_unit_beta_no_decay_retrieves_v():
    """d = 1, beta = 1: S'^T k = ||k||^2 v + (1 - ||k||^2) S^T k  (~ v)."""
    w = tiny(dk=8, rank=16, lower_bound=0.0)

    def mutate(inp):
        inp["beta"] = torch.full_like(inp["beta"], float("inf"))

    _, o = prepare(w, mutate)
    res = oracle.run(o, mode="f64", want_intermediates=True)
    for r in range(w.batch):
        sel = resolve(o, r)
        if sel is None:
            continue
        for h in range(w.heads):
            k = tb.l2_normalise(f64(res["inter"][r, h, 0, 1]))
            v = f64(res["inter"][r, h, 0, 2])
            S0 = o["state"][sel[0], h].astype(np.float64)      # [i][j]
            S1 = res["state"][sel[0], h].astype(np.float64)
            kk = float(k @ k)
            want = kk * v + (1 - kk) * (S0 @ k)
            np.testing.assert_allclose(S1 @ k, want, rtol=1e-6, atol=1e-6)
            np.testing.assert_allclose(S1 @ k, v, rtol=1e-4, atol=1e-4)


# ------------------------------------------------------------ epilogue (a10)

def test_gated_rmsnorm_matches_textbook():
    w = tiny(dk=16, rank=16, tokens=2, slot_layout="verify", conv_width=4,
             num_slots=8)
    _, o = prepare(w)
    res = oracle.run(o, mode="f64", want_intermediates=True)
    D, H, T = w.dk, w.heads, w.tokens
    for r in range(w.batch):
        if resolve(o, r) is None:
            continue
        for h in range(H):
            for t in range(T):
                ob = f64(tb.rne_bf16_bits(res["o"][r, h, t]))
                want = tb.gated_rmsnorm(ob, f64(o["norm_weight"]),
                                        f64(o["gate"][r * T + t, h * D:(h + 1) * D]),
                                        float(np.float32(o["eps"])))
                got = res["output"][r * T + t, h * D:(h + 1) * D]
                assert bf16_ulp_diff(got, tb.rne_bf16_bits(want)).max() <= 1


def test_rmsnorm_unit_gate_unit_weight_has_unit_rms():
    w = tiny(dk=32, rank=16, batch=2, heads=2)

    def mutate(inp):
        inp["gate"] = torch.full_like(inp["gate"], float("inf"))
        inp["norm_weight"] = torch.ones_like(inp["norm_weight"])

    _, o = prepare(w, mutate)
    res = oracle.run(o, mode="f32", want_intermediates=True)
    eps = float(np.float32(o["eps"]))
    for r in range(w.batch):
        if resolve(o, r) is None:
            continue
        for h in range(w.heads):
            y = f64(res["output"][r, h * w.dk:(h + 1) * w.dk])
            m = np.mean(f64(tb.rne_bf16_bits(res["o"][r, h, 0])) ** 2)
            # RMS(out) = sqrt(m / (m + eps)): 1 up to eps and BF16 rounding
            want = np.sqrt(m / (m + eps))
            assert abs(np.sqrt(np.mean(y * y)) - want) < 1e-2


# ----------------------------------------------- slots, padding, verify (a1, a7, a9)

def test_padding_writes_zeros_and_touches_nothing():
    w = tiny(batch=5, pad=2, num_slots=8)

    def sentinel(inp):
        inp["state"] = torch.full_like(inp["state"], float("nan"))
        inp["conv_state"] = torch.full_like(inp["conv_state"], float("nan"))
        inp["slots"] = torch.tensor([0, 3, -1, 0, 5], dtype=torch.int32)

    inp, o = prepare(w, sentinel)
    # live requests read real pages
    o["state"][3] = 0.25
    o["state"][5] = -0.5
    o["conv_state"][[3, 5]] = f32_to_bf16_bits(np.ones(1))[0]
    before_state = o["state"].copy()
    before_conv = o["conv_state"].copy()
    res = oracle.run(o, mode="f32")
    D, H = w.dk, w.heads
    for r in (0, 2, 3):
        assert not res["output"][r].any()            # +0.0 BF16 everywhere
    pad_pages = [s for s in range(w.num_slots) if s not in (3, 5)]
    assert np.array_equal(res["state"][pad_pages].view(np.uint32),
                          before_state[pad_pages].view(np.uint32))
    assert np.array_equal(res["conv_state"][pad_pages], before_conv[pad_pages])
    assert res["err"] == 0
    assert np.isfinite(f64(res["output"][[1, 4]])).all()


def test_out_of_range_indices_raise_error_flags_and_pad():
    w = tiny(tokens=3, slot_layout="verify", conv_width=5, num_slots=13, batch=4)
    inp, o = prepare(w)
    o["slots"] = np.array([[1, 2, 3], [4, 99, 5], [6, 7, 8], [9, 10, 11]], np.int32)
    o["accepted"] = np.array([1, 2, 0, 3], np.int32)
    res = oracle.run(o, mode="f32")
    assert res["err"] == oracle.ERR_SLOT | oracle.ERR_ACCEPTED
    assert not res["output"][1 * 3:2 * 3].any()       # slot 99 -> error item
    assert not res["output"][2 * 3:3 * 3].any()       # accepted 0 -> error item
    assert res["output"][0:3].any() and res["output"][9:12].any()


def test_verify_equals_chained_decodes():
    T = 3
    wv = tiny(tokens=T, slot_layout="verify", conv_width=T + 2, num_slots=3 * T + 1,
              dk=16, rank=16)
    _, ov = prepare(wv)
    ver = oracle.run(ov, mode="f32")
    B, H, D = wv.batch, wv.heads, wv.dk
    dim = H * D
    for r in range(B):
        a = int(ov["accepted"][r])
        src = int(ov["slots"][r, a - 1])
        cs = int(ov["slots"][r, 0])
        # decode pools: slot 1 holds the item's page, conv columns a-1..a+1
        od = dict(ov)
        od.update(batch=1, tokens=1, slot_cols=1, conv_width=3, num_slots=2,
                  accepted=None)
        state = np.zeros((2, H, D, D), np.float32)
        state[1] = ov["state"][src]
        conv = np.zeros((2, 3 * dim, 3), np.uint16)
        conv[1] = ov["conv_state"][cs][:, a - 1:a + 2]
        for t in range(T):
            row = r * T + t
            od.update(x=ov["x"][row:row + 1], f_a=ov["f_a"][row:row + 1],
                      beta=ov["beta"][row:row + 1], gate=ov["gate"][row:row + 1],
                      slots=np.array([1], np.int32), state=state, conv_state=conv)
            dec = oracle.run(od, mode="f32")
            state, conv = dec["state"], dec["conv_state"]
            assert np.array_equal(dec["output"][0], ver["output"][row])
            tgt = int(ov["slots"][r, t])
            assert np.array_equal(state[1], ver["state"][tgt])
        assert np.array_equal(conv[1], ver["conv_state"][cs][:, T - 1:T + 2])


def test_slot_relabelling_moves_pages_only():
    w = tiny(batch=4, num_slots=9)
    _, o = prepare(w)
    perm = np.concatenate([[0], 1 + np.random.default_rng(3).permutation(8)])
    o2 = dict(o)
    o2["state"] = np.empty_like(o["state"])
    o2["conv_state"] = np.empty_like(o["conv_state"])
    o2["state"][perm] = o["state"]
    o2["conv_state"][perm] = o["conv_state"]
    o2["slots"] = perm[o["slots"]].astype(np.int32)
    a = oracle.run(o, mode="f32")
    b = oracle.run(o2, mode="f32")
    assert np.array_equal(a["output"], b["output"])
    assert np.array_equal(b["state"][perm], a["state"])
    assert np.array_equal(b["conv_state"][perm], a["conv_state"])


# ------------------------------------------------ modes and teacher forcing

def test_teacher_forcing_with_own_intermediates_is_identity():
    w = tiny(dk=16, rank=16, tokens=2, slot_layout="verify", conv_width=4,
             num_slots=8)
    _, o = prepare(w)
    a = oracle.run(o, mode="f32", want_intermediates=True)
    b = oracle.run(o, mode="f32", forced=a["inter"])
    for k in ("output", "state", "conv_state"):
        assert np.array_equal(a[k], b[k])


def test_f32_and_f64_modes_agree_under_shared_intermediates():
    w = Workload("small128", batch=3, heads=2, tokens=2, num_slots=7,
                 conv_width=4, slot_layout="verify", seed=11)
    _, o = prepare(w)
    a = oracle.run(o, mode="f32", want_intermediates=True)
    b = oracle.run(o, mode="f64", forced=a["inter"])
    np.testing.assert_allclose(a["state"], b["state"], rtol=1e-4, atol=1e-5)
    assert bf16_ulp_diff(a["output"], b["output"]).max() <= 2


def test_static_argument_validation():
    w = tiny()
    _, o = prepare(w)
    for bad in (dict(tokens=0), dict(tokens=9), dict(gate_mode=2), dict(record=1)):
        with pytest.raises(ValueError):
            oracle.run(dict(o, **bad), mode="f32")


# ------------------------------------------------------------ record replay

@pytest.mark.parametrize("tokens", [2, 5])
def test_record_replay_reproduces_per_token_states(tokens):
    """Record verify + replay of a accepted tokens == the state a non-record
    verify writes after token a-1, bit for bit (same FP32 operations)."""
    T = tokens
    w = tiny(dk=8, rank=16, tokens=T, slot_layout="verify", conv_width=T + 2,
             num_slots=3 * T + 4, batch=3, heads=2, gate_mode=1, has_bias=True)
    _, o = prepare(w)
    B, H = w.batch, w.heads
    # non-record verify: per-token states in slots[r, t]
    ver = oracle.run(o, mode="f32")
    # record verify of the same step: checkpoint slot = slots[r, accepted-1]
    orec = dict(o, record=1)
    rec = oracle.run(orec, mode="f32")
    assert np.array_equal(rec["state"], o["state"])
    for a in range(0, T + 1):
        src = np.array([o["slots"][r, int(o["accepted"][r]) - 1] for r in range(B)],
                       np.int32)
        used = set(int(x) for x in o["slots"].ravel())
        free = [x for x in range(1, w.num_slots) if x not in used]
        dst = np.array(free[:B], np.int32)
        st, err = oracle.recover(state=o["state"], src_slots=src, dst_slots=dst,
                                 accepted=np.full(B, a, np.int32),
                                 rec_u=rec["rec_u"], rec_kg=rec["rec_kg"],
                                 a_log=o["a_log"], dt_bias=o["dt_bias"],
                                 lower_bound=o["lower_bound"])
        assert err == 0
        for r in range(B):
            if src[r] <= 0:
                continue
            for h in range(H):
                want = (o["state"][src[r], h] if a == 0 else
                        ver["state"][int(o["slots"][r, a - 1]), h])
                assert np.array_equal(st[dst[r], h].view(np.uint32),
                                      want.view(np.uint32)), (a, r, h)


def test_record_replay_padding_and_errors():
    T = 3
    w = tiny(dk=8, rank=16, tokens=T, slot_layout="verify", conv_width=T + 2,
             num_slots=12, batch=3, heads=2)
    _, o = prepare(w)
    rec = oracle.run(dict(o, record=1), mode="f32")
    before = o["state"].copy()
    st, err = oracle.recover(state=before, src_slots=[0, 2, 99], dst_slots=[5, 0, 6],
                             accepted=[1, 2, 1], rec_u=rec["rec_u"],
                             rec_kg=rec["rec_kg"], a_log=o["a_log"],
                             dt_bias=o["dt_bias"], lower_bound=o["lower_bound"])
    assert err == oracle.ERR_SLOT
    assert np.array_equal(st, before)          # padding rows and the error row write nothing
    st, err = oracle.recover(state=before, src_slots=[1, 2, 3], dst_slots=[4, 5, 6],
                             accepted=[1, 9, 0], rec_u=rec["rec_u"],
                             rec_kg=rec["rec_kg"], a_log=o["a_log"],
                             dt_bias=o["dt_bias"], lower_bound=o["lower_bound"])
    assert err == oracle.ERR_ACCEPTED
    assert np.array_equal(st[6], before[3])     # accepted 0 copies the checkpoint
    assert np.array_equal(st[5], before[5])     # the bad row wrote nothing


# ------------------------------------------------------------ FP32 conv state

def test_fp32_conv_state_holding_bf16_values_matches_bf16_pool():
    T = 3
    w = tiny(dk=8, rank=16, tokens=T, slot_layout="verify", conv_width=T + 3,
             num_slots=12, has_bias=True)
    _, o = prepare(w)
    o32 = dict(o, conv_state=f64(o["conv_state"]).astype(np.float32))
    a = oracle.run(o, mode="f32")
    b = oracle.run(o32, mode="f32")
    for k in ("output", "state"):
        assert np.array_equal(a[k], b[k])
    assert np.array_equal(f64(a["conv_state"]).astype(np.float32), b["conv_state"])


def test_fp32_conv_state_uses_unrounded_taps():
    T = 2
    w = tiny(tokens=T, slot_layout="verify", conv_width=T + 2, num_slots=10,
             conv_dtype="f32")
    _, o = prepare(w)
    assert o["conv_state"].dtype == np.float32
    res = oracle.run(o, mode="f64", want_intermediates=True)
    D, H = w.dk, w.heads
    for r in range(w.batch):
        sel = resolve(o, r)
        if sel is None:
            continue
        s, cs, off = sel
        for h in range(H):
            for part in range(3):
                for c in range(D):
                    ch = part * H * D + h * D + c
                    taps = o["conv_state"][cs, ch, off:off + 3].astype(np.float64)
                    xs = f64(o["x"][r * T:(r + 1) * T, ch])
                    wt = f64(o["conv_weight"][part, :, h * D + c])
                    y = tb.silu(tb.causal_conv4(taps, xs, wt))
                    np.testing.assert_allclose(res["pre"][r, h, :, part, c], y,
                                               rtol=1e-13, atol=1e-15)
            # window written as FP32: [tap1, tap2, x_0 .. x_{T-1}]
            ch = np.arange(3 * H * D).reshape(3, H, D)[:, h, :].ravel()
            new = res["conv_state"][cs][ch, :T + 2]
            old = o["conv_state"][cs][ch]
            assert np.array_equal(new[:, 0], old[:, off + 1])
            assert np.array_equal(new[:, 1], old[:, off + 2])
            xcols = f64(o["x"][r * T:(r + 1) * T][:, ch]).T.astype(np.float32)
            assert np.array_equal(new[:, 2:], xcols)
