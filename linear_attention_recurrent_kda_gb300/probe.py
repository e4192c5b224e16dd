"""Binding of the measurement probe (include/kda_probe.h,
``libkda_probe_gb300.so``): the KDA step's state-page traffic with none of
its arithmetic, the bandwidth ceiling of the step's own access pattern.  A
bench instrument, loaded only by the benchmark and the tests; the product
library (``lib``) does not carry it.  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build
from . import lib as _lib

_P = ctypes.c_void_p
EXPORTED = ("kda_probe_page_copy",)


class KdaProbeArgs(ctypes.Structure):
    """Mirror of ``struct kda_probe_args``."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("num_slots", ctypes.c_int32), ("stages", ctypes.c_int32),
        ("state", _P), ("slots", _P), ("err", _P),
        ("tokens", ctypes.c_int32), ("slot_cols", ctypes.c_int32), ("accepted", _P),
        ("sched", _P),
    ]


_probe = None


def load() -> ctypes.CDLL:
    """Load (building first if needed) the probe library."""
    global _probe
    if _probe is not None:
        return _probe
    p = _build.PROBE_LIB_PATH
    if not os.path.exists(p):
        _build.build()
    if not os.path.exists(p):
        raise ImportError(f"KDA probe library not found at {p}")
    lib = ctypes.CDLL(p)
    lib.kda_probe_page_copy.argtypes = [ctypes.POINTER(KdaProbeArgs), ctypes.c_void_p]
    lib.kda_probe_page_copy.restype = ctypes.c_int
    _probe = lib
    return lib


def call(args: KdaProbeArgs, stream_handle: int) -> int:
    """Raw call: returns the library's code without raising."""
    return int(load().kda_probe_page_copy(ctypes.byref(args),
                                          ctypes.c_void_p(stream_handle or None)))


def _check(name, t, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous {dtype} tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def kda_probe_page_copy(*, state, slots, accepted=None, tokens: int = 1, stages: int = 2,
                        err=None, sched=None,
                        stream: Optional[torch.cuda.Stream] = None) -> None:
    """The step's page traffic with no arithmetic.  ``state`` float32
    [num_slots, heads, 128, 128]; decode (``tokens`` 1): ``slots`` int32
    [batch], every page read and written back in place; verify (``tokens``
    T > 1): ``slots`` int32 [batch, >= T] and ``accepted`` int32 [batch], the
    page at slot ``slots[r, accepted[r]-1]`` written to each ``slots[r, t]``.
    ``sched`` (int32 [2], zero): the step's schedule of shared items."""
    _check("state", state, torch.float32)
    if state.dim() != 4 or tuple(state.shape[2:]) != (128, 128):
        raise ValueError("state must be [num_slots, heads, 128, 128]")
    _check("slots", slots, torch.int32)
    T = int(tokens)
    if T == 1:
        if slots.dim() == 2 and slots.shape[1] == 1:
            slots = slots.view(-1)
        if slots.dim() != 1:
            raise ValueError("slots must be [batch] for tokens == 1")
        cols = 1
    else:
        if slots.dim() != 2 or slots.shape[1] < T:
            raise ValueError("slots must be [batch, >= tokens]")
        _check("accepted", accepted, torch.int32, (slots.shape[0],))
        cols = slots.shape[1]
    if sched is not None:
        _check("sched", sched, torch.int32, (2,))
    for name, t in (("slots", slots), ("accepted", accepted), ("err", err), ("sched", sched)):
        if t is not None and t.device != state.device:
            raise ValueError(f"{name} is on {t.device}, state on {state.device}")
    a = KdaProbeArgs()
    a.batch, a.heads, a.num_slots, a.stages = (slots.shape[0], state.shape[1],
                                               state.shape[0], int(stages))
    a.tokens, a.slot_cols = T, cols
    a.state, a.slots = state.data_ptr(), slots.data_ptr()
    a.accepted = accepted.data_ptr() if T > 1 else None
    a.err = err.data_ptr() if err is not None else None
    a.sched = sched.data_ptr() if sched is not None else None
    with torch.cuda.device(state.device):
        s = stream if stream is not None else torch.cuda.current_stream(state.device)
        rc = call(a, s.cuda_stream)
    if rc != _lib.KDA_SUCCESS:
        raise _lib.KdaError(rc, _lib.strerror(rc))
