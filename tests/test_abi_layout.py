"""The ctypes mirrors of the C-ABI structs match the headers field by field:
the same names in the same order, the same kinds (32-bit integer, float,
pointer), and the same byte offsets and sizes as the C compiler lays them
out (a small C program built with gcc against include/ prints them).  A
struct changed in a header without its mirror (or the reverse) fails here
on the CPU, before any call could read a field at the wrong offset."""
from __future__ import annotations

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from linear_attention_recurrent_kda_gb300 import lib as kl
from linear_attention_recurrent_kda_gb300 import probe as kp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BUILD = os.path.join(ROOT, "tests", "_build")

STRUCTS = [
    ("kda.h", "kda_args", kl.KdaArgs),
    ("kda.h", "kda_recover_args", kl.KdaRecoverArgs),
    ("kda.h", "kda_oproj_args", kl.KdaOprojArgs),
    ("kda_probe.h", "kda_probe_args", kp.KdaProbeArgs),
]


def header_fields(header, name):
    """(field, kind) of `typedef struct name { ... } name;` in declaration
    order; kind is 'i32', 'f32' or 'ptr'."""
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    m = re.search(r"typedef\s+struct\s+%s\s*\{(.*?)\}\s*%s\s*;" % (name, name), text, flags=re.S)
    assert m, f"struct {name} not found in {header}"
    out = []
    for decl in m.group(1).split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        base = re.match(r"(?:const\s+)?(int32_t|float|void)\b", decl)
        assert base, f"unexpected declaration in {name}: {decl!r}"
        rest = decl[base.end():]
        for d in rest.split(","):
            d = d.strip()
            ptr = "*" in d
            field = d.replace("*", "").strip()
            kind = "ptr" if ptr else {"int32_t": "i32", "float": "f32"}[base.group(1)]
            out.append((field, kind))
    return out


def ctypes_fields(cls):
    kinds = {ctypes.c_int32: "i32", ctypes.c_float: "f32", ctypes.c_void_p: "ptr"}
    return [(n, kinds[t]) for n, t in cls._fields_]


@pytest.mark.parametrize("header,name,cls", STRUCTS, ids=[s[1] for s in STRUCTS])
def test_mirror_names_and_kinds(header, name, cls):
    assert ctypes_fields(cls) == header_fields(header, name)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_offsets_and_sizes_match_the_c_compiler():
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(BUILD, "abi_layout.c")
    exe = os.path.join(BUILD, "abi_layout")
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "kda_probe.h"',
             "int main(void) {"]
    for header, name, cls in STRUCTS:
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in header_fields(header, name):
            lines.append(f'  printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    with open(src, "w") as f:
        f.write("\n".join(lines) + "\n")
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                   check=True, capture_output=True)
    got = {}
    for line in subprocess.run([exe], check=True, capture_output=True,
                               text=True).stdout.splitlines():
        *key, val = line.split()
        got[tuple(key)] = int(val)
    for header, name, cls in STRUCTS:
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for field, _ in header_fields(header, name):
            assert got[(name, field)] == getattr(cls, field).offset, f"{name}.{field}"
