"""In-tree build of the native libraries (no GPU needed: nvcc cross-compiles).

* ``libwan_attn.so``  - the CUDA library behind ``include/wan_attn.h``,
  compiled for sm_103a only, with the CUDA runtime linked statically.
* ``libwan_synth.so`` - the seeded input generator (plain C, OpenMP).

Usage: ``python -m long_sequence_attention_02_b300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")

ATTN_SOURCES = ["api.cu", "rope.cu", "rows.cu", "attn_fwd.cu", "attn_fwd_fp8.cu", "attn_bwd.cu", "conv3d.cu"]
ATTN_HEADERS = ["common.cuh", "kernels.cuh"]
ATTN_LIB = os.path.join(HERE, "libwan_attn.so")
# -DWAN_DEBUG: device-side invariant checks write the error word (WAN_ERR_DEVICE_CHECK)
ATTN_DEBUG_LIB = os.path.join(HERE, "libwan_attn_debug.so")
SYNTH_LIB = os.path.join(HERE, "libwan_synth.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_synth(force: bool = False) -> str:
    src = os.path.join(CSRC, "synth.c")
    if force or _stale(SYNTH_LIB, [src]):
        tmp = SYNTH_LIB + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, SYNTH_LIB)
    return SYNTH_LIB


def build_attn(force: bool = False, verbose_ptxas: bool = False, extra=(), debug: bool = False) -> str:
    srcs = [os.path.join(CSRC, s) for s in ATTN_SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in ATTN_HEADERS] + [os.path.join(INCLUDE, "wan_attn.h")]
    target = ATTN_DEBUG_LIB if debug else ATTN_LIB
    if debug:
        extra = (*extra, "-DWAN_DEBUG")
    if not (force or _stale(target, deps)):
        return target
    tmp = target + ".tmp"
    cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-cudart", "static", "--expt-relaxed-constexpr",
           "-I", INCLUDE, "-o", tmp, *srcs, *extra]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, target)
    return target


def build_all(force: bool = False) -> None:
    build_synth(force)
    build_attn(force)
    build_attn(force, debug=True)


if __name__ == "__main__":
    build_all(force="--force" in sys.argv)
    print(ATTN_LIB)
    print(ATTN_DEBUG_LIB)
    print(SYNTH_LIB)
