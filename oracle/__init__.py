"""CPU oracle of the KDA decode / speculative-verify step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The library under
``linear_attention_recurrent_kda_gb300`` never imports it, and it imports
nothing from there: the two sides share only the seeded input generator.

The arithmetic lives in ``kda_oracle.c`` (plain C, one scalar loop nest per
(request, head) item, restating the step of the vLLM API page
"vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide", class
KdaWide) and ``oproj_oracle.c`` (the output-projection consumer epilogue of
the page "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.oproj.consumer",
class OprojConsumer, per token).  This module compiles it with gcc (``-ffp-contract=off``, OpenMP when
available) and calls it through ctypes on numpy arrays:

* ``mode="f32"``: every elementary operation correctly rounded to FP32, the
  BF16 rounding points of the page (the reference result);
* ``mode="f64"``: the same BF16 rounding points, all else in double (used by
  the pins to bound the FP32 rounding of the f32 mode).

BF16 arrays are passed as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_SRC_OPROJ = os.path.join(_HERE, "oproj_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")

ERR_SLOT = 1
ERR_ACCEPTED = 2

_P = ctypes.c_void_p


class _Args(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("tokens", ctypes.c_int32), ("dk", ctypes.c_int32),
        ("rank", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("conv_width", ctypes.c_int32), ("slot_cols", ctypes.c_int32),
        ("gate_mode", ctypes.c_int32), ("has_bias", ctypes.c_int32),
        ("record", ctypes.c_int32),
        ("x", _P), ("conv_weight", _P), ("conv_bias", _P), ("f_a", _P),
        ("f_b", _P), ("beta", _P), ("gate", _P), ("norm_weight", _P),
        ("a_log", _P), ("dt_bias", _P),
        ("slots", _P), ("accepted", _P),
        ("conv_state", _P), ("state", _P), ("output", _P),
        ("rec_u", _P), ("rec_kg", _P),
        ("lower_bound", ctypes.c_float), ("scale", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("items", _P), ("n_items", ctypes.c_int32),
        ("inter_out", _P), ("pre_out", _P), ("inter_in", _P), ("o_out", _P),
        ("err", _P), ("threads", ctypes.c_int32),
        ("conv_f32", ctypes.c_int32), ("conv_state_f32", _P),
        ("silu_in_out", _P),
    ]


class _RecoverArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("tokens", ctypes.c_int32), ("dk", ctypes.c_int32),
        ("num_slots", ctypes.c_int32),
        ("src_slots", _P), ("dst_slots", _P), ("accepted", _P),
        ("rec_u", _P), ("rec_kg", _P), ("a_log", _P), ("dt_bias", _P),
        ("lower_bound", ctypes.c_float), ("state", _P), ("err", _P),
        ("threads", ctypes.c_int32),
    ]


class _OprojArgs(ctypes.Structure):
    _fields_ = [
        ("tp", ctypes.c_int32), ("tokens", ctypes.c_int32),
        ("hidden", ctypes.c_int32), ("nb", ctypes.c_int32),
        ("has_delta", ctypes.c_int32),
        ("partials", _P), ("blocks", _P), ("norm", _P), ("query", _P),
        ("out_norm", _P), ("prefix", _P), ("output", _P),
        ("eps", ctypes.c_float), ("out_eps", ctypes.c_float),
        ("prefix_in", _P), ("pre_out", _P), ("out_pre", _P),
        ("threads", ctypes.c_int32),
    ]


def _compile(out_path: str) -> None:
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    base = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-ffp-contract=off",
            "-fno-fast-math"]
    with tempfile.TemporaryDirectory(dir=_BUILD) as tmp:
        for omp in (["-fopenmp"], []):
            objs = []
            ok = True
            for src, macro in ((_SRC, "KDA_ORACLE_F64"), (_SRC_OPROJ, "KDA_OPROJ_F64")):
                for f64 in (0, 1):
                    stem = os.path.splitext(os.path.basename(src))[0]
                    obj = os.path.join(tmp, f"{stem}_f{64 if f64 else 32}.o")
                    cmd = base + omp + [f"-D{macro}={f64}", "-c", src, "-o", obj]
                    if subprocess.run(cmd, capture_output=True).returncode != 0:
                        ok = False
                        break
                    objs.append(obj)
                if not ok:
                    break
            if not ok:
                continue
            tmp_so = os.path.join(tmp, "lib.so")
            link = ["gcc", "-shared"] + omp + objs + ["-lm", "-o", tmp_so]
            if subprocess.run(link, capture_output=True).returncode == 0:
                os.replace(tmp_so, out_path)
                return
    raise RuntimeError("could not compile the KDA oracle with gcc")


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` and ``oproj_oracle.c`` into
    ``oracle/_build/libkda_oracle.so``."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                  os.path.getmtime(_SRC_OPROJ)))
    if force or stale:
        _compile(_LIB_PATH)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        for sfx in ("f32", "f64"):
            fn = getattr(lib, f"kda_oracle_step_{sfx}")
            fn.argtypes = [ctypes.POINTER(_Args)]
            fn.restype = ctypes.c_int
            rf = getattr(lib, f"kda_oracle_recover_{sfx}")
            rf.argtypes = [ctypes.POINTER(_RecoverArgs)]
            rf.restype = ctypes.c_int
            mt = getattr(lib, f"kda_oracle_max_threads_{sfx}")
            mt.restype = ctypes.c_int
            of = getattr(lib, f"kda_oracle_oproj_{sfx}")
            of.argtypes = [ctypes.POINTER(_OprojArgs)]
            of.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle uses by default (OpenMP; 1 if built without it)."""
    return int(_load().kda_oracle_max_threads_f32())


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a: Optional[np.ndarray], dtype) -> Optional[np.ndarray]:
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


STATIC_KEYS = ("batch", "heads", "tokens", "dk", "rank", "num_slots",
               "conv_width", "slot_cols", "gate_mode", "has_bias", "record")


def run(inputs: Dict[str, object], *, mode: str = "f32",
        items: Optional[Sequence[int]] = None,
        forced: Optional[np.ndarray] = None,
        want_intermediates: bool = False,
        in_place: bool = False, threads: int = 0) -> Dict[str, np.ndarray]:
    """Run the step on host arrays.

    ``inputs`` holds the static sizes (``STATIC_KEYS``), the scalars
    ``lower_bound``, ``scale``, ``eps`` and the arrays named in
    ``kda_oracle.c`` (BF16 as uint16, FP32 as float32, slots int32).
    ``state`` and ``conv_state`` are updated in a copy unless ``in_place``.
    ``items`` restricts the step to the listed (r*heads + h) items.
    ``forced`` (uint16 [batch, heads, tokens, 4, dk]) replaces the oracle's own
    BF16 q, k, v and raw gates (teacher forcing).
    Returns output, state, conv_state, rec_u, rec_kg, err and, on request,
    inter (BF16 intermediates), pre (their unrounded values), silu_in (the
    SiLU arguments of q, k, v: [batch, heads, tokens, 3, dk]) and o (the
    recurrence output before rounding).
    """
    if mode not in ("f32", "f64"):
        raise ValueError(mode)
    lib = _load()
    st = {k: int(inputs[k]) for k in STATIC_KEYS}
    B, H, T, D = st["batch"], st["heads"], st["tokens"], st["dk"]
    u16, f32, i32 = np.uint16, np.float32, np.int32
    keep = {
        "x": _c(inputs["x"], u16),
        "conv_weight": _c(inputs["conv_weight"], u16),
        "conv_bias": _c(inputs.get("conv_bias"), u16) if st["has_bias"] else None,
        "f_a": _c(inputs["f_a"], u16), "f_b": _c(inputs["f_b"], u16),
        "beta": _c(inputs["beta"], u16), "gate": _c(inputs["gate"], u16),
        "norm_weight": _c(inputs["norm_weight"], u16),
        "a_log": _c(inputs["a_log"], f32), "dt_bias": _c(inputs["dt_bias"], f32),
        "slots": _c(inputs["slots"], i32),
        "accepted": _c(inputs.get("accepted"), i32) if T > 1 else None,
    }
    state = _c(inputs["state"], f32)
    conv_f32 = np.asarray(inputs["conv_state"]).dtype == np.float32
    conv_state = _c(inputs["conv_state"], f32 if conv_f32 else u16)
    if not in_place:
        state = state.copy()
        conv_state = conv_state.copy()
    out = np.zeros((B * T, H * D), dtype=u16)
    rec_u = np.zeros((B, H, T, D), dtype=f32) if st["record"] else None
    rec_kg = np.zeros((B, H, T, 2 * D), dtype=u16) if st["record"] else None
    inter = np.zeros((B, H, T, 4, D), dtype=u16) if want_intermediates else None
    pre = np.zeros((B, H, T, 4, D), dtype=np.float64) if want_intermediates else None
    o = np.zeros((B, H, T, D), dtype=np.float64) if want_intermediates else None
    silu_in = np.zeros((B, H, T, 3, D), dtype=np.float64) if want_intermediates else None
    forced_c = _c(forced, u16) if forced is not None else None
    items_c = None if items is None else np.ascontiguousarray(items, dtype=i32)
    err = np.zeros(1, dtype=i32)

    a = _Args()
    for k in STATIC_KEYS:
        setattr(a, k, st[k])
    for k, v in keep.items():
        setattr(a, k, _ptr(v))
    a.conv_state = None if conv_f32 else _ptr(conv_state)
    a.conv_f32 = int(conv_f32)
    a.conv_state_f32 = _ptr(conv_state) if conv_f32 else None
    a.state, a.output = _ptr(state), _ptr(out)
    a.rec_u, a.rec_kg = _ptr(rec_u), _ptr(rec_kg)
    a.lower_bound = float(inputs["lower_bound"])
    a.scale = float(inputs["scale"])
    a.eps = float(inputs["eps"])
    a.items = _ptr(items_c)
    a.n_items = 0 if items_c is None else int(items_c.size)
    a.inter_out, a.pre_out, a.o_out = _ptr(inter), _ptr(pre), _ptr(o)
    a.inter_in = _ptr(forced_c)
    a.silu_in_out = _ptr(silu_in)
    a.err = _ptr(err)
    a.threads = int(threads)
    fn = getattr(lib, f"kda_oracle_step_{mode}")
    rc = fn(ctypes.byref(a))
    if rc != 0:
        raise ValueError(f"oracle rejected the static arguments {st}")
    res = {"output": out, "state": state, "conv_state": conv_state,
           "rec_u": rec_u, "rec_kg": rec_kg, "err": int(err[0])}
    if want_intermediates:
        res.update(inter=inter, pre=pre, o=o, silu_in=silu_in)
    return res


def recover(*, state: np.ndarray, src_slots, dst_slots, accepted, rec_u: np.ndarray,
            rec_kg: np.ndarray, a_log, dt_bias, lower_bound: float,
            mode: str = "f32", in_place: bool = False, threads: int = 0):
    """Record replay (see ``kda_oracle.c``): returns (state, err).

    ``rec_u`` float32 [B, H, T, dk], ``rec_kg`` uint16 [B, H, T, 2*dk]."""
    lib = _load()
    st = _c(state, np.float32)
    if not in_place:
        st = st.copy()
    B, H, T, D = rec_u.shape
    keep = dict(src=np.ascontiguousarray(src_slots, dtype=np.int32),
                dst=np.ascontiguousarray(dst_slots, dtype=np.int32),
                acc=np.ascontiguousarray(accepted, dtype=np.int32),
                ru=_c(rec_u, np.float32), rk=_c(rec_kg, np.uint16),
                al=_c(np.asarray(a_log), np.float32),
                dt=_c(np.asarray(dt_bias), np.float32))
    err = np.zeros(1, dtype=np.int32)
    a = _RecoverArgs()
    a.batch, a.heads, a.tokens, a.dk, a.num_slots = B, H, T, D, st.shape[0]
    a.src_slots, a.dst_slots, a.accepted = (_ptr(keep["src"]), _ptr(keep["dst"]),
                                            _ptr(keep["acc"]))
    a.rec_u, a.rec_kg = _ptr(keep["ru"]), _ptr(keep["rk"])
    a.a_log, a.dt_bias = _ptr(keep["al"]), _ptr(keep["dt"])
    a.lower_bound = float(lower_bound)
    a.state, a.err, a.threads = _ptr(st), _ptr(err), int(threads)
    rc = getattr(lib, f"kda_oracle_recover_{mode}")(ctypes.byref(a))
    if rc != 0:
        raise ValueError("oracle recover rejected its arguments")
    return st, int(err[0])


def oproj(*, partials: np.ndarray, prefix: np.ndarray, out_norm: np.ndarray,
          blocks: Optional[np.ndarray] = None, norm: Optional[np.ndarray] = None,
          query: Optional[np.ndarray] = None, has_delta: bool = True,
          eps: float = 1e-6, out_eps: float = 1e-6, mode: str = "f64",
          forced_prefix: Optional[np.ndarray] = None, threads: int = 0
          ) -> Dict[str, np.ndarray]:
    """Output-projection consumer epilogue (see ``oproj_oracle.c``).

    BF16 arrays as ``numpy.uint16``: ``partials`` [tp, tokens, hidden],
    ``prefix`` [tokens, hidden] (not modified: the new prefix is returned),
    ``blocks`` [tokens, nb, hidden] or None, ``norm``/``query``/``out_norm``
    [hidden].  ``forced_prefix`` replaces the oracle's own new prefix (teacher
    forcing).  Returns prefix (the new prefix), output, pre (the new prefix
    before rounding, float64) and out_pre (the output before rounding)."""
    if mode not in ("f32", "f64"):
        raise ValueError(mode)
    lib = _load()
    u16 = np.uint16
    part = _c(partials, u16)
    tp, T, D = part.shape
    nb = 0 if blocks is None else int(np.asarray(blocks).shape[1])
    blk = _c(blocks, u16) if nb else None
    nrm = _c(norm, u16) if nb else None
    qry = _c(query, u16) if nb else None
    onrm = _c(out_norm, u16)
    pref = _c(prefix, u16).copy()
    out = np.zeros((T, D), dtype=u16)
    pre = np.zeros((T, D), dtype=np.float64)
    out_pre = np.zeros((T, D), dtype=np.float64)
    forced = _c(forced_prefix, u16) if forced_prefix is not None else None
    a = _OprojArgs()
    a.tp, a.tokens, a.hidden, a.nb, a.has_delta = tp, T, D, nb, int(bool(has_delta))
    a.partials, a.blocks, a.norm, a.query = _ptr(part), _ptr(blk), _ptr(nrm), _ptr(qry)
    a.out_norm, a.prefix, a.output = _ptr(onrm), _ptr(pref), _ptr(out)
    a.eps, a.out_eps = float(eps), float(out_eps)
    a.prefix_in, a.pre_out, a.out_pre = _ptr(forced), _ptr(pre), _ptr(out_pre)
    a.threads = int(threads)
    rc = getattr(lib, f"kda_oracle_oproj_{mode}")(ctypes.byref(a))
    if rc != 0:
        raise ValueError("oracle oproj rejected its arguments")
    return {"prefix": pref, "output": out, "pre": pre, "out_pre": out_pre}
