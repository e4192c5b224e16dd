"""Algorithmic byte accounting of one KDA step (roofline numerator).

Counts every byte the step must move between HBM and the SMs once, from the
workload's sizes and slot tables; no value of the step is computed here.
"""
from __future__ import annotations

from typing import Dict

import torch

from .workloads import Workload


def step_bytes(w: Workload, inputs: Dict[str, object]) -> Dict[str, int]:
    """Algorithmic HBM bytes of one step of ``w`` (each byte the step must
    read or write once), split into state bytes and the rest.

    Live items read their 64 KiB state page once; decode writes it back once;
    verify writes it once per token whose target slot is > 0; record mode
    writes no state.  Every other operand counts once at its own size:
    per-item conv rows (read 3 columns window + write T+2 columns), x, gate,
    output; per-request f_a and beta; per-head f_b, conv weights and bias,
    dt_bias; the slot tables.
    """
    B, H, T, D, R = w.batch, w.heads, w.tokens, w.dk, w.rank
    slots = inputs["slots"]
    page = D * D * 4
    if T == 1:
        live_req = (slots > 0).view(B)
        writes_per_req = live_req.to(torch.int64)
    else:
        acc = inputs["accepted"].to(torch.int64)
        sel = slots.gather(1, (acc - 1).view(B, 1)).view(B)
        live_req = sel > 0
        if w.record:
            writes_per_req = torch.zeros(B, dtype=torch.int64)
        else:
            writes_per_req = ((slots[:, :T] > 0).sum(1)) * live_req
    live = int(live_req.sum()) * H
    state_read = live * page
    state_write = int(writes_per_req.sum()) * H * page
    conv = live * 3 * D * (3 + T + 2) * 2
    x = live * 3 * D * T * 2
    gate = live * D * T * 2
    out = B * H * D * T * 2
    fa = int(live_req.sum()) * T * R * 2 + B * T * H * 2  # f_a + beta
    per_head = H * (D * R * 2 + 3 * 4 * D * 2 + D * 4 + 4) + H * D * 2
    if w.has_bias:
        per_head += H * 3 * D * 2
    rec = live * T * (D * 4 + 2 * D * 2) if w.record else 0
    tables = slots.numel() * 4 + (B * 4 if T > 1 else 0)
    other = conv + x + gate + out + fa + per_head + rec + tables
    return {"state": state_read + state_write, "other": other,
            "total": state_read + state_write + other}


# FP32 work of one token of one live item in the recurrence (per key j and
# value row i: S *= d, S k, S += k u, S q): 16,384 multiplies + 3 x 16,384
# fused multiply-adds at 2 flop each.
RECURRENCE_FLOP_PER_TOKEN_ITEM = 128 * 128 + 3 * 128 * 128 * 2


def recurrence_flop(w: Workload, inputs: Dict[str, object]) -> int:
    """FP32 recurrence flop of one step of ``w``: live items x tokens x
    RECURRENCE_FLOP_PER_TOKEN_ITEM (padding and error items do no work)."""
    B, H, T = w.batch, w.heads, w.tokens
    slots = inputs["slots"]
    if T == 1:
        live_req = int((slots > 0).sum())
    else:
        acc = inputs["accepted"].to(torch.int64)
        ok = (acc >= 1) & (acc <= T)
        sel = slots.gather(1, (acc.clamp(1, T) - 1).view(B, 1)).view(B)
        live_req = int(((sel > 0) & ok).sum())
    return live_req * H * T * RECURRENCE_FLOP_PER_TOKEN_ITEM
