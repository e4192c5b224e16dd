"""Pins of the output-projection consumer oracle (``oracle/oproj_oracle.c``).

The oracle restates the per-token arithmetic of the vLLM API page
"vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.oproj.consumer"
(class OprojConsumer).  These checks tie it to things other than itself:

* no earlier blocks: the output is the library RMSNorm
  (``torch.nn.functional.rms_norm``) of the new prefix times out_norm;
* integer partial sums: the new prefix is the exact sum rounded to BF16 by
  torch (with a delta: prefix + rounded sum, rounded again);
* blocks all equal to the new prefix: every candidate has the same logit, the
  mix is the prefix itself, so the output equals the no-block output;
* one block aligned with the combined weight and a large query: the softmax
  is one-hot on it and the output is that block's library RMSNorm;
* a constant combined weight and one block that permutes the prefix's
  features: block and prefix tie, so the output is the library RMSNorm of
  their sum (the prefix is a softmax candidate);
* permuting the blocks changes nothing; scaling every candidate by 2 (exact
  in BF16) with eps = 0 changes nothing;
* the FP32 mode (the page's operation order) stays within FP32 rounding of
  the float64 definition (absolute against the output's RMS: the softmax
  passes the logits' absolute rounding error on), and teacher forcing
  replaces the new prefix.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle


def bf(x) -> np.ndarray:
    """float array -> BF16 bits (round to nearest even, by torch)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def val(b: np.ndarray) -> np.ndarray:
    """BF16 bits -> float64 values."""
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def inputs(seed, tp=4, T=3, D=256, nb=3):
    rng = np.random.default_rng(seed)
    return dict(
        partials=bf(rng.normal(0, 0.4, (tp, T, D))),
        prefix=bf(rng.normal(0, 1, (T, D))),
        blocks=bf(rng.normal(0, 1, (T, nb, D))) if nb else None,
        norm=bf(rng.uniform(0.5, 1.5, D)),
        query=bf(rng.normal(0, 1, D)),
        out_norm=bf(rng.uniform(0.5, 1.5, D)),
    )


def lib_rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    t = torch.from_numpy(x)
    return torch.nn.functional.rms_norm(t, (x.shape[-1],), torch.from_numpy(w),
                                        eps=eps).numpy()


def new_prefix_exact(inp, has_delta):
    s = val(inp["partials"]).sum(axis=0)          # exact for these BF16 sums
    p = val(bf(s))
    if has_delta:
        p = val(bf(val(inp["prefix"]) + p))
    return p


@pytest.mark.parametrize("has_delta", [False, True])
@pytest.mark.parametrize("mode", ["f64", "f32"])
def test_no_blocks_is_library_rmsnorm(has_delta, mode):
    inp = inputs(1, tp=5, T=4, D=512, nb=0)
    r = oracle.oproj(**inp, has_delta=has_delta, eps=1e-6, out_eps=1e-5, mode=mode)
    p = new_prefix_exact(inp, has_delta)
    assert np.array_equal(val(r["prefix"]), p)
    want = lib_rmsnorm(p, val(inp["out_norm"]), 1e-5)
    tol = 1e-12 if mode == "f64" else 2e-6
    assert np.allclose(r["out_pre"], want, rtol=tol, atol=tol)


def test_integer_partials_round_to_bf16_exactly():
    T, D, tp = 2, 64, 16
    rng = np.random.default_rng(2)
    part = rng.integers(-40, 41, (tp, T, D)).astype(np.float32)
    part[:, 0, 0] = 20.0                      # sum 320: a BF16 value
    part[:, 0, 1] = [20.0] * 15 + [21.0]      # sum 321 -> 320 (8 significant bits)
    part[:, 0, 2] = [20.0] * 15 + [22.0]      # sum 322: BF16 spacing is 2 there
    inp = dict(partials=bf(part), prefix=bf(rng.integers(-100, 100, (T, D))),
               out_norm=bf(np.ones(D)))
    for mode in ("f32", "f64"):
        for has_delta in (False, True):
            r = oracle.oproj(**inp, has_delta=has_delta, mode=mode)
            exact = part.astype(np.int64).sum(axis=0).astype(np.float64)
            p = val(bf(exact))
            if has_delta:
                p = val(bf(val(inp["prefix"]) + p))
            assert np.array_equal(val(r["prefix"]), p), (mode, has_delta)
    r = oracle.oproj(**inp, has_delta=False)
    assert val(r["prefix"])[0, :3].tolist() == [320.0, 320.0, 322.0]


def test_blocks_equal_to_the_prefix_give_the_plain_rmsnorm():
    inp = inputs(3, tp=3, T=2, D=256, nb=0)
    p_bits = bf(new_prefix_exact(inp, False))
    base = oracle.oproj(**inp, has_delta=False)
    for nb in (1, 4, 8):
        blocks = np.repeat(p_bits[:, None, :], nb, axis=1)
        r = oracle.oproj(**{**inp, "blocks": blocks, "norm": bf(np.ones(256) * 0.7),
                            "query": bf(np.linspace(-1, 1, 256))}, has_delta=False)
        assert np.allclose(r["out_pre"], base["out_pre"], rtol=1e-12, atol=1e-12), nb


def test_a_dominant_block_takes_the_output():
    D, T, nb = 256, 2, 5
    inp = inputs(4, tp=2, T=T, D=D, nb=nb)
    norm = val(inp["norm"])
    query = val(inp["query"]) * 64.0
    w = norm * val(bf(query))
    blocks = val(inp["blocks"]).copy()
    star = 3
    blocks[:, star, :] = w / np.sqrt(np.mean(w * w))   # aligned with w, RMS 1
    inp.update(query=bf(query), blocks=bf(blocks))
    r = oracle.oproj(**inp, has_delta=False)
    want = lib_rmsnorm(val(inp["blocks"])[:, star, :], val(inp["out_norm"]), 1e-6)
    assert np.allclose(r["out_pre"], want, rtol=1e-6, atol=1e-6)


def test_the_prefix_is_a_softmax_candidate():
    D, T = 256, 3
    inp = inputs(10, tp=3, T=T, D=D, nb=0)
    p = new_prefix_exact(inp, False)
    perm = np.random.default_rng(11).permutation(D)
    blocks = bf(p[:, perm])[:, None, :]          # same sum and RMS as p
    r = oracle.oproj(**{**inp, "blocks": blocks, "norm": bf(np.full(D, 0.75)),
                        "query": bf(np.full(D, 1.5))}, has_delta=False)
    want = lib_rmsnorm(p + p[:, perm], val(inp["out_norm"]), 1e-6 * 4)
    assert np.allclose(r["out_pre"], want, rtol=1e-9, atol=1e-9)


def test_block_order_does_not_matter():
    inp = inputs(5, tp=4, T=3, D=384, nb=6)
    r0 = oracle.oproj(**inp)
    perm = np.array([4, 1, 5, 0, 3, 2])
    r1 = oracle.oproj(**{**inp, "blocks": inp["blocks"][:, perm, :]})
    assert np.array_equal(r0["prefix"], r1["prefix"])
    assert np.allclose(r0["out_pre"], r1["out_pre"], rtol=1e-12, atol=1e-14)


def test_scaling_every_candidate_changes_nothing():
    inp = inputs(6, tp=4, T=2, D=256, nb=4)
    r0 = oracle.oproj(**inp, has_delta=False, eps=0.0, out_eps=0.0)
    twice = {**inp, "partials": bf(val(inp["partials"]) * 2.0),
             "blocks": bf(val(inp["blocks"]) * 2.0)}
    r1 = oracle.oproj(**twice, has_delta=False, eps=0.0, out_eps=0.0)
    assert np.array_equal(val(r1["prefix"]), 2.0 * val(r0["prefix"]))
    assert np.allclose(r1["out_pre"], r0["out_pre"], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("nb,tp", [(0, 16), (1, 1), (8, 16), (3, 7)])
def test_fp32_order_stays_within_rounding_of_the_definition(nb, tp):
    inp = inputs(7 + nb, tp=tp, T=4, D=1024, nb=nb)
    r64 = oracle.oproj(**inp, mode="f64")
    r32 = oracle.oproj(**inp, mode="f32", forced_prefix=r64["prefix"])
    # Block logits reach |35| here; a sequential FP32 sum over 1024 features
    # leaves ~1e-4 of absolute error in them, which moves the softmax weights
    # by the same relative amount.  Elements where two weighted blocks nearly
    # cancel then carry that error against the output's RMS (about 1), not
    # against their own size: the bound is absolute at 2e-4 of the RMS.
    err = np.abs(r32["out_pre"] - r64["out_pre"])
    rms = np.sqrt(np.mean(r64["out_pre"] ** 2, axis=1, keepdims=True))
    assert np.all(err <= 2e-4 * rms + 1e-5 * np.abs(r64["out_pre"]))
    # the new prefix: equal unless the exact value sits at a BF16 midpoint
    own = oracle.oproj(**inp, mode="f32")
    diff = own["prefix"] != r64["prefix"]
    assert diff.mean() < 1e-3


def test_teacher_forcing_replaces_the_new_prefix():
    inp = inputs(9, tp=4, T=2, D=128, nb=2)
    forced = bf(np.full((2, 128), 0.5))
    r = oracle.oproj(**inp, forced_prefix=forced)
    assert np.array_equal(r["prefix"], forced)
    inp2 = dict(inp, blocks=None)
    r2 = oracle.oproj(**inp2, forced_prefix=forced)
    want = lib_rmsnorm(np.full((2, 128), 0.5), val(inp["out_norm"]), 1e-6)
    assert np.allclose(r2["out_pre"], want, rtol=1e-12, atol=1e-12)
