"""Roofline numerators of the bench (host logic, no GPU): the algorithmic
bytes and the FP32 recurrence flop of each workload, checked against the
sizes written out by hand from the workload tables."""
from __future__ import annotations

from linear_attention_recurrent_kda_gb300.accounting import (
    RECURRENCE_FLOP_PER_TOKEN_ITEM, recurrence_flop, step_bytes)
from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, make_inputs

PAGE = 128 * 128 * 4


def test_flop_per_token_item():
    # S *= d (16,384 multiplies) and three multiply-add sweeps (S k, S += k u, S q).
    assert RECURRENCE_FLOP_PER_TOKEN_ITEM == 114_688


def test_decode_b256_h32():
    w = WORKLOADS["decode_b256_h32"]
    inp = make_inputs(w)
    b = step_bytes(w, inp)
    assert b["state"] == 8192 * 2 * PAGE            # every page read and written once
    assert 0 < b["other"] < 0.06 * b["state"]
    assert recurrence_flop(w, inp) == 8192 * 114_688


def test_padded_decode_counts_live_items_only():
    w = WORKLOADS["decode_b64_h32_pad8"]
    inp = make_inputs(w)
    live = int((inp["slots"] > 0).sum()) * w.heads
    assert live == 56 * 32
    assert step_bytes(w, inp)["state"] == live * 2 * PAGE
    assert recurrence_flop(w, inp) == live * 114_688


def test_verify_q4_writes_one_page_per_token():
    w = WORKLOADS["verify_q4_b128_h32"]
    inp = make_inputs(w)
    assert step_bytes(w, inp)["state"] == 4096 * PAGE + 4096 * 4 * PAGE
    assert recurrence_flop(w, inp) == 4096 * 4 * 114_688


def test_record_q8_reads_pages_and_writes_records():
    w = WORKLOADS["verify_q8_record_b64_h64"]
    inp = make_inputs(w)
    live = 58 * 64                                      # 6 of 64 requests padded
    b = step_bytes(w, inp)
    assert b["state"] == live * PAGE                    # no state write in record mode
    assert b["other"] >= live * 8 * (128 * 4 + 256 * 2)  # the records
    assert recurrence_flop(w, inp) == live * 8 * 114_688
