"""Host-side conversions shared by the tests: torch CPU tensors from the seeded
input generator -> numpy arrays the oracle takes (BF16 as uint16 bits), and
BF16 bit helpers used by the comparisons.  No step arithmetic lives here."""
from __future__ import annotations

from typing import Dict

import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> uint16 bit pattern (numpy); other dtypes -> numpy."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_oracle(inputs: Dict[str, object]) -> Dict[str, object]:
    out = {}
    for k, v in inputs.items():
        out[k] = bits(v) if isinstance(v, torch.Tensor) else v
    return out


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round FP32 values to BF16 (nearest-even) through torch."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_ordinal(b: np.ndarray) -> np.ndarray:
    """Monotone integer index of BF16 bit patterns (so |a-b| counts ulps)."""
    b = b.astype(np.int64)
    neg = (b & 0x8000) != 0
    mag = b & 0x7FFF
    return np.where(neg, -mag, mag)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(bf16_ordinal(a) - bf16_ordinal(b))
