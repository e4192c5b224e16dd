"""Build the in-tree CUDA library ``libkda_gb300.so`` for sm_103a.

The translation units of csrc/ (the step, split, replay, output-projection,
self-test and probe kernels) compiled by nvcc in parallel with a single
``-gencode arch=compute_103a,code=sm_103a`` and linked into one shared
library, which sits next to this file and is loaded by
``linear_attention_recurrent_kda_gb300.lib``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(HERE, "libkda_gb300.so")
SOURCES = [os.path.join(CSRC, n) for n in ("kda_step.cu", "kda_split.cu",
                                            "kda_recover.cu", "kda_oproj.cu",
                                            "kda_selftest.cu", "kda_probe.cu")]
HEADERS = [os.path.join(INCLUDE, "kda.h"), os.path.join(CSRC, "kda_device.cuh")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > t for s in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if missing or older than its sources.

    Each translation unit compiles in its own nvcc process (in parallel), then
    one nvcc call links the shared library."""
    if not force and not is_stale():
        return LIB_PATH
    with tempfile.TemporaryDirectory() as tmp:
        procs = []
        objs = []
        for src in SOURCES:
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            cmd = [nvcc()] + NVCC_FLAGS + ["-I", INCLUDE, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
            objs.append(obj)
        logs = []
        for src, pr in procs:
            out, _ = pr.communicate()
            logs.append(out)
            if pr.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{out}")
        out = os.path.join(tmp, "libkda_gb300.so")
        link = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                "-o", out] + objs
        res = subprocess.run(link, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
        if verbose:
            print("".join(logs))
        os.replace(out, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
