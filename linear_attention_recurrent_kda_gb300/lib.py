"""ctypes view of the C ABI in include/kda.h (``libkda_gb300.so``).

Argument marshalling only: every step of the KDA decode/verify path runs in
the CUDA library.  Loading fails loudly when the library is missing; there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

_P = ctypes.c_void_p

# Return codes and device error flags (include/kda.h).
KDA_SUCCESS = 0
KDA_ERR_NULL_ARGS = 1
KDA_ERR_TOKENS = 2
KDA_ERR_GATE_MODE = 3
KDA_ERR_RECORD = 4
KDA_ERR_NULL_POINTER = 5
KDA_ERR_CONV_WIDTH = 6
KDA_ERR_ALIGNMENT = 7
KDA_ERR_SHAPE = 8
KDA_ERR_DEVICE = 9
KDA_ERR_LAUNCH = 10
KDA_ERR_PATH = 11
KDA_PATH_AUTO, KDA_PATH_PERSISTENT, KDA_PATH_SPLIT = 0, 1, 2
KDA_DEVERR_SLOT = 1
KDA_DEVERR_ACCEPTED = 2
KDA_DEVERR_TIMEOUT = 4

EXPORTED = ("kda_decode", "kda_verify", "kda_step_noalloc", "kda_recover", "kda_oproj",
            "kda_selftest_wait_timeout", "kda_strerror", "kda_abi_version")


class KdaArgs(ctypes.Structure):
    """Mirror of ``struct kda_args``."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("tokens", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("conv_width", ctypes.c_int32), ("slot_cols", ctypes.c_int32),
        ("gate_mode", ctypes.c_int32), ("has_bias", ctypes.c_int32),
        ("record", ctypes.c_int32), ("use_pdl", ctypes.c_int32),
        ("x", _P), ("conv_weight", _P), ("conv_bias", _P), ("f_a", _P),
        ("f_b", _P), ("beta", _P), ("gate", _P), ("norm_weight", _P),
        ("a_log", _P), ("dt_bias", _P), ("slots", _P), ("accepted", _P),
        ("conv_state", _P), ("state", _P), ("output", _P),
        ("rec_u", _P), ("rec_kg", _P),
        ("lower_bound", ctypes.c_float), ("scale", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("err", _P), ("dbg", _P), ("path", ctypes.c_int32),
        ("conv_f32", ctypes.c_int32), ("sched", _P),
    ]


class KdaRecoverArgs(ctypes.Structure):
    """Mirror of ``struct kda_recover_args``."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("tokens", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("src_slots", _P), ("dst_slots", _P), ("accepted", _P),
        ("rec_u", _P), ("rec_kg", _P), ("a_log", _P), ("dt_bias", _P),
        ("lower_bound", ctypes.c_float), ("state", _P), ("err", _P), ("sched", _P),
    ]


class KdaOprojArgs(ctypes.Structure):
    """Mirror of ``struct kda_oproj_args``."""
    _fields_ = [
        ("tp", ctypes.c_int32), ("tokens", ctypes.c_int32),
        ("hidden", ctypes.c_int32), ("nb", ctypes.c_int32),
        ("has_delta", ctypes.c_int32),
        ("partials", _P), ("blocks", _P), ("norm", _P), ("query", _P),
        ("out_norm", _P), ("prefix", _P), ("output", _P),
        ("eps", ctypes.c_float), ("out_eps", ctypes.c_float),
    ]


class KdaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"KDA error {code}: {msg}")
        self.code = code


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if path is None and not os.path.exists(p):
        _build.build()
    if not os.path.exists(p):
        raise ImportError(f"KDA CUDA library not found at {p}")
    lib = ctypes.CDLL(p)
    for name in ("kda_decode", "kda_verify", "kda_step_noalloc"):
        fn = getattr(lib, name)
        fn.argtypes = [ctypes.POINTER(KdaArgs), ctypes.c_void_p]
        fn.restype = ctypes.c_int
    lib.kda_recover.argtypes = [ctypes.POINTER(KdaRecoverArgs), ctypes.c_void_p]
    lib.kda_recover.restype = ctypes.c_int
    lib.kda_oproj.argtypes = [ctypes.POINTER(KdaOprojArgs), ctypes.c_void_p]
    lib.kda_oproj.restype = ctypes.c_int
    lib.kda_selftest_wait_timeout.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.kda_selftest_wait_timeout.restype = ctypes.c_int
    lib.kda_strerror.argtypes = [ctypes.c_int]
    lib.kda_strerror.restype = ctypes.c_char_p
    lib.kda_abi_version.argtypes = []
    lib.kda_abi_version.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().kda_strerror(int(code)).decode()


def call(entry: str, args, stream_handle: int) -> int:
    """Raw call: returns the library's code without raising."""
    fn = getattr(load(), entry)
    return int(fn(ctypes.byref(args), ctypes.c_void_p(stream_handle or None)))
