"""Failure detection and out-of-bounds guards on the GPU (no fault involved).

* The bounded on-chip wait (the one every kernel uses) runs out on a barrier
  that nothing completes, raises KDA_DEVERR_TIMEOUT in the error word, and
  the context afterwards runs a step that still matches the oracle.
* Guard rows filled with a NaN bit pattern directly before and after the
  state pool, the conv pool, the output and the record buffers stay
  bit-identical through decode, verify (with error and padding items) and
  record steps on both kernel paths, and the results equal an unguarded run.
"""
from __future__ import annotations

import ctypes
import time

import numpy as np
import pytest
import torch

from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300.api import step_from_inputs
from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, Workload, make_inputs
from tests.parity import compare, run_gpu, to_device

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_stays_usable():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    t0 = time.time()
    rc = kl.load().kda_selftest_wait_timeout(ctypes.c_void_p(err.data_ptr()),
                                             ctypes.c_void_p(stream.cuda_stream))
    assert rc == kl.KDA_SUCCESS
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert int(err.item()) == kl.KDA_DEVERR_TIMEOUT
    assert 1.0 < waited < 30.0, waited
    inp = make_inputs(WORKLOADS["decode_b4_h8"])
    compare(inp, run_gpu(inp))


def _guarded(t: torch.Tensor, pattern: int):
    """A copy of `t` inside a buffer with one guard row before and after."""
    big = torch.empty((t.shape[0] + 2,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    ib = big.view(torch.int16 if t.element_size() == 2 else torch.int32)
    ib.fill_(pattern)
    big[1:-1].copy_(t)
    return big, big[1:-1]


NAN16 = 0x7FC1            # a BF16 NaN with a payload
NAN32 = 0x7FC00001        # an FP32 NaN with a payload


def _guard_ok(big: torch.Tensor, pattern: int) -> bool:
    ib = big.view(torch.int16 if big.element_size() == 2 else torch.int32)
    want = torch.full_like(ib[0], pattern)
    return bool(torch.equal(ib[0], want) and torch.equal(ib[-1], want))


def run_guarded(inp, path):
    d = to_device(inp)
    B, H, T = d["batch"], d["heads"], d["tokens"]
    bigs = {}
    for k in ("state", "conv_state"):
        pat = NAN32 if d[k].dtype == torch.float32 else NAN16
        big, d[k] = _guarded(d[k], pat)
        bigs[k] = (big, pat)
    out_big, out = _guarded(torch.full((B * T, H * 128), float("nan"), dtype=torch.bfloat16,
                                       device="cuda"), NAN16)
    bigs["output"] = (out_big, NAN16)
    ru = rk = None
    if d["record"]:
        ru_big, ru = _guarded(torch.zeros((B, H, T, 128), dtype=torch.float32,
                                          device="cuda"), NAN32)
        rk_big, rk = _guarded(torch.zeros((B, H, T, 256), dtype=torch.bfloat16,
                                          device="cuda"), NAN16)
        bigs["rec_u"], bigs["rec_kg"] = (ru_big, NAN32), (rk_big, NAN16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step_from_inputs(d, out, rec_u=ru, rec_kg=rk, err=err, path=path)()
    torch.cuda.synchronize()
    for k, (big, pat) in bigs.items():
        assert _guard_ok(big, pat), f"guard rows of {k} changed"
    res = {"output": out.cpu(), "state": d["state"].cpu(), "conv_state": d["conv_state"].cpu(),
           "err": int(err.item())}
    if d["record"]:
        res.update(rec_u=ru.cpu(), rec_kg=rk.cpu())
    return res


def plain(inp, path):
    d = to_device(inp)
    B, H, T = d["batch"], d["heads"], d["tokens"]
    out = torch.full((B * T, H * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ru = rk = None
    if d["record"]:
        ru = torch.zeros((B, H, T, 128), dtype=torch.float32, device="cuda")
        rk = torch.zeros((B, H, T, 256), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step_from_inputs(d, out, rec_u=ru, rec_kg=rk, err=err, path=path)()
    torch.cuda.synchronize()
    res = {"output": out.cpu(), "state": d["state"].cpu(), "conv_state": d["conv_state"].cpu(),
           "err": int(err.item())}
    if d["record"]:
        res.update(rec_u=ru.cpu(), rec_kg=rk.cpu())
    return res


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    ia = a.view(torch.int16 if a.element_size() == 2 else torch.int32)
    ib = b.view(torch.int16 if b.element_size() == 2 else torch.int32)
    return bool(torch.equal(ia, ib))


CASES = {
    "decode_pad": Workload("g_dec", batch=9, heads=4, tokens=1, num_slots=20, conv_width=3,
                           slot_layout="decode", pad=2, seed=301),
    "verify_errors": Workload("g_ver", batch=7, heads=3, tokens=4, num_slots=7 * 4 + 3,
                              conv_width=6, slot_layout="verify", pad=1, seed=302),
    "record": Workload("g_rec", batch=6, heads=4, tokens=8, num_slots=9, conv_width=10,
                       slot_layout="checkpoint", pad=1, gate_mode=1, has_bias=True,
                       record=True, seed=303),
}


@pytest.mark.parametrize("path", [kl.KDA_PATH_PERSISTENT, kl.KDA_PATH_SPLIT])
@pytest.mark.parametrize("case", sorted(CASES))
def test_guard_rows_untouched_and_results_unchanged(case, path):
    inp = make_inputs(CASES[case])
    if case == "verify_errors":
        inp["slots"][2, 1] = 10_000          # write target beyond the pool
        inp["accepted"][4] = 0               # accepted out of range
        inp["slots"][5, 0] = -1              # live item without a conv slot
        inp["accepted"][5] = 2
    g = run_guarded(inp, path)
    p = plain(inp, path)
    assert g["err"] == p["err"]
    for k in p:
        if k != "err":
            assert _same(g[k], p[k]), k
