"""Seeded synthetic inputs for the KDA decode / speculative-verify step.

This module only draws random numbers and lays out slot tables.  It holds none
of the step's arithmetic, so both the CUDA library's tests/benchmark and the
CPU oracle can take their inputs from it.

All draws use a CPU ``torch.Generator`` seeded per workload, in a fixed order,
so the GPU path and the oracle read identical bytes.  BF16 tensors are drawn in
FP32 and rounded to nearest-even by torch.  Distributions (std dev, not
variance, for every N(0, s)):

====================  ===================================================
x                     N(0, 1) BF16 [B*T, 3*H*dk]   (q | k | v blocks)
conv_state            N(0, 1) BF16 (or FP32) [num_slots, 3*H*dk, conv_width]
conv_weight           N(0, 0.5) BF16 [3, 4, H*dk]
conv_bias             N(0, 0.5) BF16 [3*H*dk]      (has_bias only)
f_a                   N(0, 1) BF16 [B*T, rank]
f_b                   N(0, 0.1) BF16 [H*dk, rank]  (feature, rank)
a_log                 U(-1, 1) FP32 [H]
dt_bias               N(0, 0.1) FP32 [H*dk]
beta                  N(0, 1) BF16 [B*T, H]        raw logits
state                 N(0, 0.1) FP32 [num_slots, H, dk, dk]
gate                  N(0, 1) BF16 [B*T, H*dk]
norm_weight           U(0.5, 1.5) BF16 [dk]
lower_bound, scale    -5, dk**-0.5;  eps 1e-6
====================  ===================================================

Slot tables (slot 0 is the null slot, ``slot <= 0`` marks padding):

* ``decode``:     B distinct slots drawn from 1..num_slots-1; ``pad`` of them
                  set to 0.
* ``verify``:     [B, T] distinct per-token slots from 1..num_slots-1;
                  ``pad`` request rows set to 0; accepted ~ U{1..T}.
* ``checkpoint``: one distinct slot per request repeated across its T columns
                  (record mode reads and never writes the state); ``pad``
                  request rows set to 0; accepted ~ U{1..T}.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    tokens: int
    num_slots: int
    conv_width: int
    slot_layout: str  # "decode" | "verify" | "checkpoint"
    pad: int = 0
    gate_mode: int = 0
    has_bias: bool = False
    record: bool = False
    dk: int = 128
    rank: int = 128
    seed: int = 1000
    lower_bound: float = -5.0
    eps: float = 1e-6
    conv_dtype: str = "bf16"  # "bf16" | "f32": element type of the conv pool

    @property
    def dim(self) -> int:
        return self.heads * self.dk

    @property
    def items(self) -> int:
        return self.batch * self.heads

    @property
    def slot_cols(self) -> int:
        return 1 if self.tokens == 1 else self.tokens

    @property
    def scale(self) -> float:
        return self.dk ** -0.5

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the KDA decode/verify benchmark description, by name.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("decode_b4_h8", batch=4, heads=8, tokens=1, num_slots=16,
                 conv_width=3, slot_layout="decode", seed=1000),
        Workload("decode_b64_h32_pad8", batch=64, heads=32, tokens=1,
                 num_slots=128, conv_width=3, slot_layout="decode", pad=8,
                 seed=1001),
        Workload("decode_b256_h32", batch=256, heads=32, tokens=1,
                 num_slots=512, conv_width=3, slot_layout="decode", seed=1002),
        Workload("verify_q4_b128_h32", batch=128, heads=32, tokens=4,
                 num_slots=4 * 128 + 1, conv_width=6, slot_layout="verify",
                 seed=1003),
        Workload("verify_q8_record_b64_h64", batch=64, heads=64, tokens=8,
                 num_slots=65, conv_width=10, slot_layout="checkpoint", pad=6,
                 gate_mode=1, has_bias=True, record=True, seed=1004),
    )
}


def _bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16)


def make_inputs(w: Workload) -> Dict[str, object]:
    """Draw every input of one step of ``w`` as CPU tensors.

    Returns a dict with the tensors, the static sizes and the scalars; the
    pools (``state``, ``conv_state``) are the step's in/out buffers.
    """
    g = torch.Generator().manual_seed(w.seed)
    B, H, T, D, R = w.batch, w.heads, w.tokens, w.dk, w.rank
    dim = H * D
    rows = B * T

    def randn(*shape, std=1.0):
        return torch.randn(*shape, generator=g) * std

    out: Dict[str, object] = {}
    out["x"] = _bf16(randn(rows, 3 * dim))
    conv = randn(w.num_slots, 3 * dim, w.conv_width)
    out["conv_state"] = conv if w.conv_dtype == "f32" else _bf16(conv)
    out["conv_weight"] = _bf16(randn(3, 4, dim, std=0.5))
    out["conv_bias"] = _bf16(randn(3 * dim, std=0.5)) if w.has_bias else None
    out["f_a"] = _bf16(randn(rows, R))
    out["f_b"] = _bf16(randn(dim, R, std=0.1))
    out["a_log"] = torch.rand(H, generator=g) * 2.0 - 1.0
    out["dt_bias"] = randn(dim, std=0.1)
    out["beta"] = _bf16(randn(rows, H))
    out["state"] = randn(w.num_slots, H, D, D, std=0.1)
    out["gate"] = _bf16(randn(rows, dim))
    out["norm_weight"] = _bf16(torch.rand(D, generator=g) + 0.5)

    free = torch.randperm(w.num_slots - 1, generator=g) + 1  # 1..num_slots-1
    if w.slot_layout == "decode":
        if B > w.num_slots - 1:
            raise ValueError("pool too small for distinct slots")
        slots = free[:B].clone()
        if w.pad:
            slots[torch.randperm(B, generator=g)[: w.pad]] = 0
        accepted = None
    elif w.slot_layout == "verify":
        if B * T > w.num_slots - 1:
            raise ValueError("pool too small for distinct per-token slots")
        slots = free[: B * T].clone().view(B, T)
        if w.pad:
            slots[torch.randperm(B, generator=g)[: w.pad]] = 0
        accepted = torch.randint(1, T + 1, (B,), generator=g)
    elif w.slot_layout == "checkpoint":
        if B > w.num_slots - 1:
            raise ValueError("pool too small for distinct checkpoint slots")
        slots = free[:B].clone().view(B, 1).repeat(1, T)
        if w.pad:
            slots[torch.randperm(B, generator=g)[: w.pad]] = 0
        accepted = torch.randint(1, T + 1, (B,), generator=g)
    else:
        raise ValueError(w.slot_layout)
    out["slots"] = slots.to(torch.int32).contiguous()
    out["accepted"] = None if accepted is None else accepted.to(torch.int32)

    out.update(
        batch=B, heads=H, tokens=T, dk=D, rank=R, num_slots=w.num_slots,
        conv_width=w.conv_width, slot_cols=w.slot_cols, gate_mode=w.gate_mode,
        has_bias=int(w.has_bias), record=int(w.record),
        lower_bound=w.lower_bound, scale=w.scale, eps=w.eps,
    )
    return out


# ------------------------------------------- output-projection consumer epilogue

@dataclass(frozen=True)
class OprojWorkload:
    """Inputs of the output-projection consumer epilogue (``kda_oproj``).

    Draws (std dev): partials N(0, 0.25) BF16 [tp, tokens, hidden] (a sum of 16
    is about N(0, 1)); prefix N(0, 1) BF16 [tokens, hidden]; blocks N(0, 1)
    BF16 [tokens, nb, hidden]; norm U(0.5, 1.5); query N(0, 3/sqrt(hidden)) so
    that block logits spread over a few units; out_norm U(0.5, 1.5); eps and
    out_eps 1e-6.
    """
    name: str
    tp: int
    tokens: int
    hidden: int
    nb: int
    has_delta: bool = True
    seed: int = 2000
    eps: float = 1e-6
    out_eps: float = 1e-6


OPROJ_WORKLOADS: Dict[str, OprojWorkload] = {
    w.name: w
    for w in (
        # The page's TP16 consumer at the decode batch of 256 rows.
        OprojWorkload("oproj_tp16_t256_h7168_nb8", tp=16, tokens=256, hidden=7168,
                      nb=8, seed=2000),
    )
}


def make_oproj_inputs(w: OprojWorkload) -> Dict[str, object]:
    """Draw the inputs of one ``kda_oproj`` call as CPU tensors."""
    g = torch.Generator().manual_seed(w.seed)

    def randn(*shape, std=1.0):
        return torch.randn(*shape, generator=g) * std

    out: Dict[str, object] = {}
    out["partials"] = _bf16(randn(w.tp, w.tokens, w.hidden, std=0.25))
    out["prefix"] = _bf16(randn(w.tokens, w.hidden))
    out["blocks"] = _bf16(randn(w.tokens, w.nb, w.hidden)) if w.nb else None
    out["norm"] = _bf16(torch.rand(w.hidden, generator=g) + 0.5) if w.nb else None
    out["query"] = _bf16(randn(w.hidden, std=3.0 / w.hidden ** 0.5)) if w.nb else None
    out["out_norm"] = _bf16(torch.rand(w.hidden, generator=g) + 0.5)
    out.update(has_delta=bool(w.has_delta), eps=w.eps, out_eps=w.out_eps)
    return out
