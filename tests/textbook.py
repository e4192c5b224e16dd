"""Float64 textbook formulations used to pin the oracle.

Each function states a step of the KDA decode/verify method in a form that
differs from the oracle's scalar loops: the logistic function through tanh,
the depthwise convolution as a sliding-window matrix product, the L2 norm
through numpy's norm, and the gated delta rule in its matrix form

    S_t = (I - beta k k^T) diag(d) S_{t-1} + beta k v^T,      o_t = S_t^T q

with S indexed [key j][value i] (the transpose of the state page layout).
"""
from __future__ import annotations

import numpy as np
from numpy.lib.stride_tricks import sliding_window_view


def sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def causal_conv4(taps: np.ndarray, xs: np.ndarray, w: np.ndarray, bias=0.0):
    """Output t = sum_i w[i] * window[t + i], window = taps (3) ++ xs (T)."""
    win = np.concatenate([np.asarray(taps, np.float64), np.asarray(xs, np.float64)])
    return sliding_window_view(win, 4) @ np.asarray(w, np.float64) + bias


def decay(a_log, raw_g, dt_bias, lower_bound):
    return np.exp(lower_bound * sigmoid(np.exp(a_log) * (raw_g + dt_bias)))


def l2_normalise(v, scale=1.0, eps=1e-6):
    v = np.asarray(v, np.float64)
    n = np.linalg.norm(v)
    return v * (scale / np.sqrt(n * n + eps))


def delta_rule(S_ji: np.ndarray, d, k, v, beta):
    """One gated delta-rule token in matrix form; returns (S_new, u).

    u = beta * (v - (diag(d) S)^T k) is the per-value-row correction the
    record mode stores."""
    D = S_ji.shape[0]
    decayed = np.diag(d) @ S_ji
    A = np.eye(D) - beta * np.outer(k, k)
    S_new = A @ decayed + beta * np.outer(k, v)
    u = beta * (v - decayed.T @ k)
    return S_new, u


def gated_rmsnorm(o, norm_weight, gate, eps):
    o = np.asarray(o, np.float64)
    return o / np.sqrt(np.mean(o * o) + eps) * norm_weight * sigmoid(gate)


def rne_bf16_bits(v) -> np.ndarray:
    """Nearest BF16 (ties to even) of float64 values, as uint16 bits.

    Takes the two BF16 neighbours (truncation towards zero of the float32
    bit pattern and its successor in magnitude) and keeps the nearer one;
    the differences are exact by Sterbenz's lemma."""
    v = np.asarray(v, np.float64).ravel()
    out = np.empty(v.size, np.uint16)
    for n, x in enumerate(v):
        if np.isnan(x):
            out[n] = 0x7FC0
            continue
        f = np.float32(x)
        if np.isinf(f):
            out[n] = 0x7F80 | (0x8000 if x < 0 else 0)
            continue
        b = int(np.array(f).view(np.uint32)) >> 16
        lo = b
        hi = b + 1
        vl = float(np.array(lo << 16, np.uint32).view(np.float32))
        vh = float(np.array((hi & 0xFFFF) << 16, np.uint32).view(np.float32))
        # float32 rounding may have crossed lo; step down when needed.
        if abs(vl) > abs(x):
            lo, hi = b - 1, b
            vh = vl
            vl = float(np.array((lo & 0xFFFF) << 16, np.uint32).view(np.float32))
        dl, dh = abs(x - vl), abs(vh - x)
        if dl < dh or (dl == dh and lo % 2 == 0):
            out[n] = lo & 0xFFFF
        else:
            out[n] = hi & 0xFFFF
    return out
