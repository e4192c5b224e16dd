"""Build the in-tree CUDA libraries for sm_103a.

``libkda_gb300.so``: the translation units of the step and its companions
(the step, split, replay, output-projection and self-test kernels; the C ABI
of include/kda.h).  ``libkda_probe_gb300.so``: the measurement probe of
include/kda_probe.h, a bench instrument kept out of the product library.
Every translation unit is compiled by its own nvcc process, in parallel, with
a single ``-gencode arch=compute_103a,code=sm_103a``; each library is linked
by one more nvcc call and sits next to this file.
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
PROBE_LIB_PATH = os.path.join(HERE, "libkda_probe_gb300.so")
SOURCES = [os.path.join(CSRC, n) for n in ("kda_step.cu", "kda_split.cu",
                                            "kda_recover.cu", "kda_oproj.cu",
                                            "kda_selftest.cu")]
PROBE_SOURCES = [os.path.join(CSRC, "kda_probe.cu")]
HEADERS = [os.path.join(INCLUDE, "kda.h"), os.path.join(INCLUDE, "kda_probe.h"),
           os.path.join(CSRC, "kda_device.cuh"), os.path.join(CSRC, "kda_host.h")]
LIBS = ((LIB_PATH, SOURCES), (PROBE_LIB_PATH, PROBE_SOURCES))

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _stale(lib: str, sources) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in list(sources) + HEADERS)


def is_stale() -> bool:
    return any(_stale(lib, srcs) for lib, srcs in LIBS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the libraries that are missing or older than their sources.

    Each translation unit compiles in its own nvcc process (all in parallel),
    then one nvcc call per library links it.  Returns the product library's
    path."""
    todo = [(lib, srcs) for lib, srcs in LIBS if force or _stale(lib, srcs)]
    if not todo:
        return LIB_PATH
    with tempfile.TemporaryDirectory() as tmp:
        procs = []
        objs = {lib: [] for lib, _ in todo}
        for lib, srcs in todo:
            for src in srcs:
                obj = os.path.join(tmp, os.path.basename(src) + ".o")
                cmd = [nvcc()] + NVCC_FLAGS + ["-I", INCLUDE, "-c", src, "-o", obj]
                if verbose:
                    cmd.insert(1, "-Xptxas=-v")
                procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                    stderr=subprocess.STDOUT, text=True)))
                objs[lib].append(obj)
        logs = []
        for src, pr in procs:
            out, _ = pr.communicate()
            logs.append(out)
            if pr.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{out}")
        for lib, _ in todo:
            out = os.path.join(tmp, os.path.basename(lib))
            link = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                    "-o", out] + objs[lib]
            res = subprocess.run(link, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
            os.replace(out, lib)
        if verbose:
            print("".join(logs))
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
