"""The C-ABI libraries build, load and export every function their headers
declare (include/kda.h: the product library; include/kda_probe.h: the
measurement probe's own library, so that the product exports only the
step's calls); host-side argument validation answers without touching a
GPU."""
from __future__ import annotations

import os
import re

import pytest

from linear_attention_recurrent_kda_gb300 import build as kbuild
from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300 import probe as kp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kda_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_header_is_covered():
    assert sorted(f for f in os.listdir(os.path.join(ROOT, "include"))
                  if f.endswith(".h")) == ["kda.h", "kda_probe.h"]


def test_library_builds_and_exports_every_declared_symbol():
    kbuild.build()
    lib = kl.load()
    names = declared_functions("kda.h")
    assert set(kl.EXPORTED) == set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/kda.h but not exported"
    # the bench instrument is not part of the product library
    assert not hasattr(lib, "kda_probe_page_copy")


def test_probe_library_exports_its_header():
    kbuild.build()
    lib = kp.load()
    names = declared_functions("kda_probe.h")
    assert set(kp.EXPORTED) == set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/kda_probe.h but not exported"


def test_version_and_strerror():
    assert kl.load().kda_abi_version() == 7
    for code in range(0, 12):
        assert kl.strerror(code)
    assert "unknown" in kl.strerror(999)


def _args(**kw):
    a = kl.KdaArgs()
    a.batch, a.heads, a.tokens, a.num_slots, a.conv_width = 2, 1, 1, 4, 3
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_null_args():
    import ctypes
    lib = kl.load()
    assert lib.kda_decode(None, None) == kl.KDA_ERR_NULL_ARGS
    assert lib.kda_verify(None, None) == kl.KDA_ERR_NULL_ARGS
    assert lib.kda_step_noalloc(None, None) == kl.KDA_ERR_NULL_ARGS


@pytest.mark.parametrize("entry,kw,code", [
    ("kda_decode", dict(tokens=0), kl.KDA_ERR_TOKENS),
    ("kda_decode", dict(tokens=2), kl.KDA_ERR_TOKENS),
    ("kda_verify", dict(tokens=1), kl.KDA_ERR_TOKENS),
    ("kda_verify", dict(tokens=9), kl.KDA_ERR_TOKENS),
    ("kda_decode", dict(gate_mode=3), kl.KDA_ERR_GATE_MODE),
    ("kda_decode", dict(record=1), kl.KDA_ERR_RECORD),
    ("kda_decode", dict(batch=-1), kl.KDA_ERR_SHAPE),
    ("kda_decode", dict(batch=0), kl.KDA_SUCCESS),
    ("kda_decode", dict(heads=0), kl.KDA_SUCCESS),
    ("kda_decode", dict(num_slots=0), kl.KDA_ERR_SHAPE),
    ("kda_verify", dict(tokens=3, slot_cols=2, conv_width=5), kl.KDA_ERR_SHAPE),
    ("kda_decode", dict(conv_width=2), kl.KDA_ERR_CONV_WIDTH),
    ("kda_decode", {}, kl.KDA_ERR_NULL_POINTER),
    # the no-allocation entry validates exactly as kda_decode / kda_verify
    # (chosen by the token count) before it touches the library's words
    ("kda_step_noalloc", dict(tokens=0), kl.KDA_ERR_TOKENS),
    ("kda_step_noalloc", dict(tokens=9), kl.KDA_ERR_TOKENS),
    ("kda_step_noalloc", dict(gate_mode=3), kl.KDA_ERR_GATE_MODE),
    ("kda_step_noalloc", dict(record=1), kl.KDA_ERR_RECORD),
    ("kda_step_noalloc", dict(batch=0), kl.KDA_SUCCESS),
    ("kda_step_noalloc", dict(tokens=3, slot_cols=2, conv_width=5), kl.KDA_ERR_SHAPE),
    ("kda_step_noalloc", dict(tokens=4, conv_width=5, slot_cols=4), kl.KDA_ERR_CONV_WIDTH),
    ("kda_step_noalloc", {}, kl.KDA_ERR_NULL_POINTER),
])
def test_host_validation_without_gpu(entry, kw, code):
    assert kl.call(entry, _args(**kw), 0) == code


def test_alignment_rule_checked_before_any_device_call():
    a = _args()
    fake = 1 << 20
    for name in ("x", "conv_weight", "f_a", "f_b", "beta", "gate", "norm_weight",
                 "a_log", "dt_bias", "slots", "conv_state", "state", "output"):
        setattr(a, name, fake)
    a.state = fake + 4            # FP32 pool must be 16-byte aligned
    assert kl.call("kda_decode", a, 0) == kl.KDA_ERR_ALIGNMENT
    assert kl.call("kda_step_noalloc", a, 0) == kl.KDA_ERR_ALIGNMENT
    a.state = fake
    a.sched = fake + 2            # scheduler words must be 4-byte aligned
    assert kl.call("kda_decode", a, 0) == kl.KDA_ERR_ALIGNMENT


def _oargs(**kw):
    a = kl.KdaOprojArgs()
    a.tp, a.tokens, a.hidden, a.nb, a.has_delta = 16, 4, 7168, 2, 1
    fake = 1 << 20
    for n in ("partials", "blocks", "norm", "query", "out_norm", "prefix", "output"):
        setattr(a, n, fake)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(tp=0), kl.KDA_ERR_SHAPE),
    (dict(tp=65), kl.KDA_ERR_SHAPE),
    (dict(tokens=-1), kl.KDA_ERR_SHAPE),
    (dict(nb=9), kl.KDA_ERR_SHAPE),
    (dict(nb=-1), kl.KDA_ERR_SHAPE),
    (dict(hidden=7168 + 256), kl.KDA_ERR_SHAPE),
    (dict(hidden=1000), kl.KDA_ERR_SHAPE),
    (dict(hidden=0), kl.KDA_ERR_SHAPE),
    (dict(tokens=0), kl.KDA_SUCCESS),
    (dict(partials=None), kl.KDA_ERR_NULL_POINTER),
    (dict(output=None), kl.KDA_ERR_NULL_POINTER),
    (dict(blocks=None), kl.KDA_ERR_NULL_POINTER),
    (dict(nb=0, blocks=None, norm=None, query=None, prefix=(1 << 20) + 8),
     kl.KDA_ERR_ALIGNMENT),
    (dict(query=(1 << 20) + 2), kl.KDA_ERR_ALIGNMENT),
])
def test_oproj_host_validation_without_gpu(kw, code):
    assert kl.call("kda_oproj", _oargs(**kw), 0) == code
    assert kl.load().kda_oproj(None, None) == kl.KDA_ERR_NULL_ARGS


def test_selftest_host_validation_without_gpu():
    import ctypes
    lib = kl.load()
    assert lib.kda_selftest_wait_timeout(None, None) == kl.KDA_ERR_NULL_POINTER
    assert lib.kda_selftest_wait_timeout(ctypes.c_void_p((1 << 20) + 2), None) == \
        kl.KDA_ERR_ALIGNMENT


def _pargs(**kw):
    a = kp.KdaProbeArgs()
    a.batch, a.heads, a.num_slots, a.stages = 4, 2, 8, 2
    a.tokens, a.slot_cols = 1, 1
    a.state, a.slots = 1 << 20, 1 << 21
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(stages=1), kl.KDA_ERR_SHAPE),
    (dict(stages=4), kl.KDA_ERR_SHAPE),
    (dict(batch=-1), kl.KDA_ERR_SHAPE),
    (dict(num_slots=0), kl.KDA_ERR_SHAPE),
    (dict(batch=0), kl.KDA_SUCCESS),
    (dict(state=None), kl.KDA_ERR_NULL_POINTER),
    (dict(slots=None), kl.KDA_ERR_NULL_POINTER),
    (dict(state=(1 << 20) + 4), kl.KDA_ERR_ALIGNMENT),
    (dict(slots=(1 << 21) + 2), kl.KDA_ERR_ALIGNMENT),
    (dict(err=(1 << 22) + 1), kl.KDA_ERR_ALIGNMENT),
    (dict(tokens=0), kl.KDA_ERR_TOKENS),
    (dict(tokens=9, slot_cols=9), kl.KDA_ERR_TOKENS),
    (dict(slot_cols=0), kl.KDA_ERR_SHAPE),
    (dict(tokens=4, slot_cols=3, accepted=1 << 23), kl.KDA_ERR_SHAPE),
    (dict(tokens=4, slot_cols=4), kl.KDA_ERR_NULL_POINTER),
    (dict(tokens=4, slot_cols=4, accepted=(1 << 23) + 2), kl.KDA_ERR_ALIGNMENT),
])
def test_probe_host_validation_without_gpu(kw, code):
    assert kp.call(_pargs(**kw), 0) == code
    assert kp.load().kda_probe_page_copy(None, None) == kl.KDA_ERR_NULL_ARGS
