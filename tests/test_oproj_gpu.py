"""GPU parity of the output-projection consumer epilogue (``kda_oproj``).

Compared with the oracle (``oracle/oproj_oracle.c``) on the same seeded
inputs:

* the new prefix (written back in place): bit-exact against the oracle's
  FP32 mode, which sums the partials in the same rank-group order; every
  value is one FP32 add chain and two BF16 roundings;
* the output: against the float64 definition run on the GPU's new prefix
  (teacher forcing), within one BF16 ulp of max(|ref|, 2^-8) plus 3e-4 of
  the row's RMS.  The absolute term covers the FP32 rounding of the block
  logits (sums over `hidden` features), which the softmax passes on as a
  relative change of the weights; the oracle's own FP32 mode needs 2e-4
  against its float64 mode for the same reason.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.api import kda_oproj
from linear_attention_recurrent_kda_gb300.workloads import (OPROJ_WORKLOADS, OprojWorkload,
                                                            make_oproj_inputs)

pytestmark = pytest.mark.gpu


def bits(t):
    return None if t is None else t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def val(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_gpu(inp):
    dev = "cuda"
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    T, D = d["prefix"].shape
    out = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device=dev)
    kda_oproj(partials=d["partials"], prefix=d["prefix"], output=out,
              out_norm=d["out_norm"], blocks=d["blocks"], norm=d["norm"],
              query=d["query"], has_delta=d["has_delta"], eps=d["eps"],
              out_eps=d["out_eps"])
    torch.cuda.synchronize()
    return bits(d["prefix"]), bits(out)


def oracle_args(inp):
    return dict(partials=bits(inp["partials"]), prefix=bits(inp["prefix"]),
                out_norm=bits(inp["out_norm"]), blocks=bits(inp["blocks"]),
                norm=bits(inp["norm"]), query=bits(inp["query"]),
                has_delta=inp["has_delta"], eps=inp["eps"], out_eps=inp["out_eps"])


def ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check(inp):
    g_prefix, g_out = run_gpu(inp)
    args = oracle_args(inp)
    own = oracle.oproj(**args, mode="f32")
    assert np.array_equal(g_prefix, own["prefix"]), \
        f"new prefix differs in {(g_prefix != own['prefix']).sum()} elements"
    ref = oracle.oproj(**args, mode="f64", forced_prefix=g_prefix)
    r = ref["out_pre"]
    rms = np.sqrt(np.mean(r * r, axis=1, keepdims=True))
    tol = ulp_bf16(np.maximum(np.abs(r), 2.0 ** -8)) + 3e-4 * rms
    err = np.abs(val(g_out) - r)
    bad = err > tol
    assert not bad.any(), (f"{bad.sum()} outputs off; worst {err.max():.3e} "
                           f"at {np.unravel_index((err / tol).argmax(), err.shape)}")
    exact = np.mean(g_out == ref["output"])
    return exact


def w(**kw):
    base = dict(name="t", tp=16, tokens=5, hidden=1024, nb=3, has_delta=True, seed=7)
    base.update(kw)
    return OprojWorkload(**base)


@pytest.mark.parametrize("tp", [1, 3, 16, 37, 64])
def test_partial_sum_groups(tp):
    exact = check(make_oproj_inputs(w(tp=tp, seed=10 + tp)))
    assert exact > 0.97


@pytest.mark.parametrize("nb", [0, 1, 2, 5, 8])
@pytest.mark.parametrize("has_delta", [False, True])
def test_blocks_and_delta(nb, has_delta):
    exact = check(make_oproj_inputs(w(nb=nb, has_delta=has_delta, seed=30 + nb)))
    assert exact > 0.97


@pytest.mark.parametrize("hidden", [256, 2048, 7168])
def test_hidden_sizes(hidden):
    check(make_oproj_inputs(w(hidden=hidden, tokens=3, seed=50 + hidden // 256)))


def test_full_size_workload():
    """The benchmark's configuration (TP16, 256 rows, hidden 7168, 8 blocks),
    every row checked."""
    exact = check(make_oproj_inputs(OPROJ_WORKLOADS["oproj_tp16_t256_h7168_nb8"]))
    assert exact > 0.97


def test_sharp_softmax_and_large_logits():
    inp = make_oproj_inputs(w(nb=8, seed=70))
    inp["query"] = inp["query"] * 40.0          # logits of tens: near one-hot
    check(inp)


def test_zero_rows_is_a_no_op_and_runs_are_deterministic():
    inp = make_oproj_inputs(w(seed=80))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.zeros((0, 1024), dtype=torch.bfloat16, device="cuda")
    kda_oproj(partials=d["partials"][:, :0].contiguous(), prefix=d["prefix"][:0].contiguous(),
              output=out, out_norm=d["out_norm"], blocks=d["blocks"][:0].contiguous(),
              norm=d["norm"], query=d["query"], has_delta=True)
    torch.cuda.synchronize()
    a = run_gpu(inp)
    b = run_gpu(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_prefix_written_in_place_and_nothing_else():
    inp = make_oproj_inputs(w(seed=90, tokens=4))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    guard = torch.full((6, 1024), 7.0, dtype=torch.bfloat16, device="cuda")
    prefix, out = guard[1:5], torch.empty((4, 1024), dtype=torch.bfloat16, device="cuda")
    prefix.copy_(d["prefix"])
    before = [t.clone() for t in (d["partials"], d["blocks"], d["norm"], d["query"],
                                  d["out_norm"])]
    kda_oproj(partials=d["partials"], prefix=prefix, output=out, out_norm=d["out_norm"],
              blocks=d["blocks"], norm=d["norm"], query=d["query"], has_delta=True)
    torch.cuda.synchronize()
    assert torch.equal(guard[0], torch.full((1024,), 7.0, dtype=torch.bfloat16, device="cuda"))
    assert torch.equal(guard[5], torch.full((1024,), 7.0, dtype=torch.bfloat16, device="cuda"))
    for b, t in zip(before, (d["partials"], d["blocks"], d["norm"], d["query"], d["out_norm"])):
        assert torch.equal(b, t)
    own = oracle.oproj(**oracle_args(inp), mode="f32")
    assert np.array_equal(bits(prefix), own["prefix"])


def test_host_errors_launch_nothing():
    inp = make_oproj_inputs(w(seed=95))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.zeros((5, 1024), dtype=torch.bfloat16, device="cuda")
    a = kl.KdaOprojArgs()
    a.tp, a.tokens, a.hidden, a.nb, a.has_delta = 16, 5, 1024, 3, 1
    a.partials, a.blocks = d["partials"].data_ptr(), d["blocks"].data_ptr()
    a.norm, a.query, a.out_norm = (d["norm"].data_ptr(), d["query"].data_ptr(),
                                   d["out_norm"].data_ptr())
    a.prefix, a.output = d["prefix"].data_ptr(), out.data_ptr()
    a.eps = a.out_eps = 1e-6
    before = d["prefix"].clone()
    a.output = out.data_ptr() + 2
    assert kl.call("kda_oproj", a, 0) == kl.KDA_ERR_ALIGNMENT
    a.output = out.data_ptr()
    a.nb = 9
    assert kl.call("kda_oproj", a, 0) == kl.KDA_ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.equal(before, d["prefix"]) and not out.any()
