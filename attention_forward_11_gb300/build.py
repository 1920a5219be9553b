"""Builds libattn.so in-tree with nvcc for sm_103a (GB300) only.

    python -m attention_forward_11_gb300.build [--verbose]

One translation unit, one -gencode, cudart linked statically (the library
needs only the driver at run time).  The output sits beside this file.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "attn_api.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("fmha_fwd_sm103.cuh", "fmha_fwd_d256_sm103.cuh", "fmha_bwd_sm103.cuh",
                                          "fmha_bwd_d256_sm103.cuh", "unit_rates_sm103.cuh", "sm103_ptx.cuh")] + [
    os.path.join(ROOT, "include", "attn.h")]
OUT = os.path.join(PKG, "libattn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date() -> bool:
    if not os.path.exists(OUT):
        return False
    t = os.path.getmtime(OUT)
    return all(os.path.getmtime(f) <= t for f in SOURCES + HEADERS + [__file__])


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return OUT
    tmp = OUT + f".tmp.{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "static", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
           *SOURCES, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv))
