"""Builds libm2rnn.so (and the micro-benchmark) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel into ``_build/`` and linked
into ``_build/libm2rnn.so``; the CUDA runtime is linked statically so the
library has no run-time dependency beyond the driver.

``build(checked=True)`` (``python -m non_linear_matrix_gb300.build checked``)
compiles the same sources with ``-DM2RNN_CHECK=1`` into
``_build/check/libm2rnn_check.so``: every computed global-memory index is
tested against its array's extent and a violation is reported through the
device status word (M2RNN_ERR_BOUNDS) instead of being performed.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libm2rnn.so")
BUILD_CHECKED = os.path.join(BUILD, "check")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libm2rnn_check.so")
MICROBENCH = os.path.join(BUILD, "m2rnn_microbench")

SOURCES = ["m2rnn_api.cu", "m2rnn_fwd.cu", "m2rnn_bwd.cu", "m2rnn_bwd_pipe.cu", "m2rnn_decode.cu",
           "m2rnn_noalloc.cu", "m2rnn_norm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, n) for n in os.listdir(CSRC)]
    paths += [os.path.join(INCLUDE, n) for n in os.listdir(INCLUDE)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link libm2rnn.so (or, checked=True, libm2rnn_check.so);
    returns its path.  Raises on failure."""
    out_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    defs = ["-DM2RNN_CHECK=1"] if checked else []
    os.makedirs(out_dir, exist_ok=True)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH, *FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.append("-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if verbose or pr.returncode != 0:
            sys.stdout.write(out.decode(errors="replace"))
        if pr.returncode != 0:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


def build_microbench() -> str:
    """Compile the pipe-rate / step-latency micro-benchmark executable."""
    os.makedirs(BUILD, exist_ok=True)
    subprocess.run([_nvcc(), *ARCH, "-O3", "-std=c++17", "-I", CSRC,
                    os.path.join(CSRC, "m2rnn_microbench.cu"), "-o", MICROBENCH], check=True)
    return MICROBENCH


if __name__ == "__main__":
    if len(sys.argv) > 1 and sys.argv[1] == "microbench":
        print(build_microbench())
    elif len(sys.argv) > 1 and sys.argv[1] == "checked":
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked=True))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
