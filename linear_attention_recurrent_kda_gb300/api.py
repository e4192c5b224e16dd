"""Python binding of the KDA decode / verify C ABI (include/kda.h).

PyTorch is used only for device memory and streams: the functions here check
that every tensor is a contiguous CUDA tensor of the documented dtype and shape,
fill ``struct kda_args`` with raw pointers and call ``kda_decode`` /
``kda_verify`` in ``libkda_gb300.so``.  Nothing of the step is computed in
Python and there is no fallback path.

Method: vLLM API page
"vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide" (KdaWide).
"""
from __future__ import annotations

from typing import Dict, Optional

import torch

from . import lib as _lib

DK = 128


def _check(name, t, dtype, shape=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _ptr(t):
    return None if t is None else t.data_ptr()


def _same_device(dev, **tensors):
    """Every given tensor (None skipped) lives on ``dev``: the kernel would
    otherwise dereference another GPU's pointer."""
    for name, t in tensors.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, expected {dev}")


class KdaStep:
    """A prepared KDA step over fixed device tensors.

    Validates once, keeps the filled ``kda_args`` and launches with
    ``__call__(stream)``; reuse it across steps that read the same buffers
    (the tensors' contents may change between calls, their storage may not).

    ``sched``: the persistent kernel's scheduler words (int32 [2], zero before
    first use; ``kda_args.sched``).  By default the step allocates its own,
    so its launches balance the last items over the CTAs; pass a tensor to
    share one between steps launched in order on one stream, or
    ``balance=False`` for fixed contiguous ranges only (same bits).
    ``noalloc=True`` allocates nothing and calls ``kda_step_noalloc``, which
    uses the library's own words (launches through it must be ordered).
    """

    def __init__(self, *, x, conv_weight, conv_state, f_a, f_b, beta, a_log,
                 dt_bias, slots, state, output, gate, norm_weight,
                 lower_bound: float, scale: float, eps: float,
                 tokens: int = 1, accepted=None, conv_bias=None,
                 gate_mode: int = 0, record: bool = False, rec_u=None,
                 rec_kg=None, err=None, dbg=None, use_pdl: bool = False,
                 path: int = 0, sched=None, balance: bool = True,
                 noalloc: bool = False):
        bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
        T = int(tokens)
        if not 1 <= T <= 8:
            raise ValueError(f"tokens must be 1..8, got {T}")
        _check("a_log", a_log, f32)
        H = a_log.shape[0]
        dim = H * DK
        _check("output", output, bf)
        if output.dim() != 2 or output.shape[1] != dim or output.shape[0] % T:
            raise ValueError("output must be [batch*tokens, heads*128]")
        B = output.shape[0] // T
        _check("state", state, f32)
        if state.dim() != 4 or tuple(state.shape[1:]) != (H, DK, DK):
            raise ValueError("state must be [num_slots, heads, 128, 128]")
        num_slots = state.shape[0]
        if not isinstance(conv_state, torch.Tensor) or conv_state.dtype not in (bf, f32):
            raise TypeError("conv_state must be a bfloat16 or float32 tensor")
        _check("conv_state", conv_state, conv_state.dtype)
        if conv_state.dim() != 3 or tuple(conv_state.shape[:2]) != (num_slots, 3 * dim):
            raise ValueError("conv_state must be [num_slots, 3*heads*128, width]")
        W = conv_state.shape[2]
        _check("x", x, bf, (B * T, 3 * dim))
        _check("conv_weight", conv_weight, bf, (3, 4, dim))
        _check("conv_bias", conv_bias, bf, (3 * dim,), allow_none=True)
        _check("f_a", f_a, bf, (B * T, DK))
        _check("f_b", f_b, bf, (dim, DK))
        _check("beta", beta, bf, (B * T, H))
        _check("dt_bias", dt_bias, f32, (dim,))
        _check("gate", gate, bf, (B * T, dim))
        _check("norm_weight", norm_weight, bf, (DK,))
        _check("slots", slots, i32)
        if T == 1:
            if slots.numel() != B:
                raise ValueError("decode slots must be [batch]")
            slot_cols = 1
        else:
            if slots.dim() != 2 or slots.shape[0] != B:
                raise ValueError("verify slots must be [batch, >= tokens]")
            slot_cols = slots.shape[1]
            _check("accepted", accepted, i32, (B,))
        if record:
            _check("rec_u", rec_u, f32, (B, H, T, DK))
            _check("rec_kg", rec_kg, bf, (B, H, T, 2 * DK))
        _check("err", err, i32, allow_none=True)
        _check("dbg", dbg, bf, (B, H, T, 4, DK), allow_none=True)
        dev = output.device
        if noalloc:
            sched = None
        elif sched is None and balance:
            sched = torch.zeros(2, dtype=i32, device=dev)
        _check("sched", sched, i32, (2,), allow_none=True)
        _same_device(dev, x=x, conv_weight=conv_weight, conv_bias=conv_bias,
                     conv_state=conv_state, f_a=f_a, f_b=f_b, beta=beta, a_log=a_log,
                     dt_bias=dt_bias, slots=slots, state=state, gate=gate,
                     norm_weight=norm_weight, accepted=accepted if T > 1 else None,
                     rec_u=rec_u if record else None, rec_kg=rec_kg if record else None,
                     err=err, dbg=dbg, sched=sched)

        a = _lib.KdaArgs()
        a.batch, a.heads, a.tokens = B, H, T
        a.num_slots, a.conv_width, a.slot_cols = num_slots, W, slot_cols
        a.gate_mode, a.has_bias = int(gate_mode), int(conv_bias is not None)
        a.record, a.use_pdl = int(bool(record)), int(bool(use_pdl))
        a.x, a.conv_weight, a.conv_bias = _ptr(x), _ptr(conv_weight), _ptr(conv_bias)
        a.f_a, a.f_b, a.beta = _ptr(f_a), _ptr(f_b), _ptr(beta)
        a.gate, a.norm_weight = _ptr(gate), _ptr(norm_weight)
        a.a_log, a.dt_bias = _ptr(a_log), _ptr(dt_bias)
        a.slots, a.accepted = _ptr(slots), _ptr(accepted if T > 1 else None)
        a.conv_state, a.state, a.output = _ptr(conv_state), _ptr(state), _ptr(output)
        a.rec_u, a.rec_kg = _ptr(rec_u), _ptr(rec_kg)
        a.lower_bound, a.scale, a.eps = float(lower_bound), float(scale), float(eps)
        a.err, a.dbg = _ptr(err), _ptr(dbg)
        a.path = int(path)
        a.conv_f32 = int(conv_state.dtype == f32)
        a.sched = _ptr(sched)
        self.args = a
        self.entry = ("kda_step_noalloc" if noalloc else
                      "kda_decode" if T == 1 else "kda_verify")
        self.device = dev
        # keep the tensors alive as long as the prepared step
        self._keep = (x, conv_weight, conv_state, f_a, f_b, beta, a_log, dt_bias,
                      slots, state, output, gate, norm_weight, accepted,
                      conv_bias, rec_u, rec_kg, err, dbg, sched)

    def __call__(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        # the library launches on the current device: make it the tensors' one
        with torch.cuda.device(self.device):
            s = stream if stream is not None else torch.cuda.current_stream(self.device)
            rc = _lib.call(self.entry, self.args, s.cuda_stream)
        if rc != _lib.KDA_SUCCESS:
            raise _lib.KdaError(rc, _lib.strerror(rc))


def kda_decode(stream: Optional[torch.cuda.Stream] = None, **kw) -> None:
    """One decode step (tokens = 1) on ``stream``; see ``KdaStep``."""
    if kw.get("tokens", 1) != 1:
        raise ValueError("kda_decode takes tokens = 1")
    KdaStep(**kw)(stream)


def kda_verify(stream: Optional[torch.cuda.Stream] = None, **kw) -> None:
    """One speculative-verify step (tokens 2..8, optional record mode)."""
    if kw.get("tokens", 1) < 2:
        raise ValueError("kda_verify takes tokens >= 2")
    KdaStep(**kw)(stream)


INPUT_KEYS = ("x", "conv_weight", "conv_bias", "conv_state", "f_a", "f_b", "beta",
              "a_log", "dt_bias", "slots", "accepted", "state", "gate",
              "norm_weight")


def step_from_inputs(dev_inputs: Dict[str, object], output: torch.Tensor, *,
                     rec_u=None, rec_kg=None, err=None, dbg=None,
                     use_pdl: bool = False, path: int = 0, sched=None,
                     balance: bool = True, noalloc: bool = False) -> KdaStep:
    """A ``KdaStep`` from a device copy of a seeded workload's input dict."""
    d = dev_inputs
    T = int(d["tokens"])
    return KdaStep(
        x=d["x"], conv_weight=d["conv_weight"], conv_state=d["conv_state"],
        f_a=d["f_a"], f_b=d["f_b"], beta=d["beta"], a_log=d["a_log"],
        dt_bias=d["dt_bias"], slots=d["slots"], state=d["state"], output=output,
        gate=d["gate"], norm_weight=d["norm_weight"],
        lower_bound=d["lower_bound"], scale=d["scale"], eps=d["eps"], tokens=T,
        accepted=d.get("accepted") if T > 1 else None,
        conv_bias=d.get("conv_bias") if d.get("has_bias") else None,
        gate_mode=int(d["gate_mode"]), record=bool(d["record"]), rec_u=rec_u,
        rec_kg=rec_kg, err=err, dbg=dbg, use_pdl=use_pdl, path=path, sched=sched,
        balance=balance, noalloc=noalloc)


def kda_recover(*, state, src_slots, dst_slots, accepted, rec_u, rec_kg, a_log,
                dt_bias, lower_bound: float, err=None, sched=None, balance: bool = True,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """Record replay (include/kda.h ``kda_recover``): rebuild the accepted
    state pages from checkpoint pages and a record-mode verify's records.
    ``sched``: scheduler words (int32 [2], zero); by default a fresh pair per
    call (``balance=False``: contiguous item ranges only, same bits)."""
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    _check("rec_u", rec_u, f32)
    if rec_u.dim() != 4 or rec_u.shape[3] != DK:
        raise ValueError("rec_u must be [batch, heads, tokens, 128]")
    B, H, T = rec_u.shape[:3]
    _check("rec_kg", rec_kg, bf, (B, H, T, 2 * DK))
    _check("state", state, f32)
    if state.dim() != 4 or tuple(state.shape[1:]) != (H, DK, DK):
        raise ValueError("state must be [num_slots, heads, 128, 128]")
    for n, t in (("src_slots", src_slots), ("dst_slots", dst_slots),
                 ("accepted", accepted)):
        _check(n, t, i32, (B,))
    _check("a_log", a_log, f32, (H,))
    _check("dt_bias", dt_bias, f32, (H * DK,))
    _check("err", err, i32, allow_none=True)
    if sched is None and balance:
        sched = torch.zeros(2, dtype=i32, device=state.device)
    _check("sched", sched, i32, (2,), allow_none=True)
    _same_device(state.device, src_slots=src_slots, dst_slots=dst_slots, accepted=accepted,
                 rec_u=rec_u, rec_kg=rec_kg, a_log=a_log, dt_bias=dt_bias, err=err,
                 sched=sched)
    a = _lib.KdaRecoverArgs()
    a.batch, a.heads, a.tokens, a.num_slots = B, H, T, state.shape[0]
    a.src_slots, a.dst_slots, a.accepted = (_ptr(src_slots), _ptr(dst_slots),
                                            _ptr(accepted))
    a.rec_u, a.rec_kg = _ptr(rec_u), _ptr(rec_kg)
    a.a_log, a.dt_bias = _ptr(a_log), _ptr(dt_bias)
    a.lower_bound = float(lower_bound)
    a.state, a.err = _ptr(state), _ptr(err)
    a.sched = _ptr(sched)
    with torch.cuda.device(state.device):
        s = stream if stream is not None else torch.cuda.current_stream(state.device)
        rc = _lib.call("kda_recover", a, s.cuda_stream)
    if rc != _lib.KDA_SUCCESS:
        raise _lib.KdaError(rc, _lib.strerror(rc))


def kda_oproj(*, partials, prefix, output, out_norm, blocks=None, norm=None,
              query=None, has_delta: bool = True, eps: float = 1e-6,
              out_eps: float = 1e-6,
              stream: Optional[torch.cuda.Stream] = None) -> None:
    """Output-projection consumer epilogue (include/kda.h ``kda_oproj``).

    ``partials`` bf16 [tp, tokens, hidden]; ``prefix`` bf16 [tokens, hidden]
    (replaced by the new prefix); ``output`` bf16 [tokens, hidden];
    ``out_norm`` bf16 [hidden]; ``blocks`` bf16 [tokens, nb, hidden] with
    ``norm``/``query`` bf16 [hidden], or None for no earlier blocks."""
    bf = torch.bfloat16
    _check("partials", partials, bf)
    if partials.dim() != 3:
        raise ValueError("partials must be [tp, tokens, hidden]")
    tp, T, D = partials.shape
    _check("prefix", prefix, bf, (T, D))
    _check("output", output, bf, (T, D))
    _check("out_norm", out_norm, bf, (D,))
    nb = 0
    if blocks is not None:
        _check("blocks", blocks, bf)
        if blocks.dim() != 3 or blocks.shape[0] != T or blocks.shape[2] != D:
            raise ValueError("blocks must be [tokens, nb, hidden]")
        nb = blocks.shape[1]
        _check("norm", norm, bf, (D,))
        _check("query", query, bf, (D,))
    _same_device(partials.device, prefix=prefix, output=output, out_norm=out_norm,
                 blocks=blocks if nb else None, norm=norm if nb else None,
                 query=query if nb else None)
    a = _lib.KdaOprojArgs()
    a.tp, a.tokens, a.hidden, a.nb = tp, T, D, nb
    a.has_delta = int(bool(has_delta))
    a.partials, a.prefix, a.output = _ptr(partials), _ptr(prefix), _ptr(output)
    a.out_norm = _ptr(out_norm)
    a.blocks = _ptr(blocks) if nb else None
    a.norm = _ptr(norm) if nb else None
    a.query = _ptr(query) if nb else None
    a.eps, a.out_eps = float(eps), float(out_eps)
    with torch.cuda.device(partials.device):
        s = stream if stream is not None else torch.cuda.current_stream(partials.device)
        rc = _lib.call("kda_oproj", a, s.cuda_stream)
    if rc != _lib.KDA_SUCCESS:
        raise _lib.KdaError(rc, _lib.strerror(rc))
