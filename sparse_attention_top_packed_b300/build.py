"""Builds the library in-tree with nvcc for sm_103a: libtopk_packed.so, and
libtopk_packed_checked.so, the same source compiled with TOPK_CHECKED (every
computed global-memory address and every shared-memory index that is not in
range by construction checked at run time; a violation is recorded in the
diagnostics word and the access skipped).  The two are compiled in parallel.

    python -m sparse_attention_top_packed_b300.build [--verbose-ptxas]
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "topk_packed.cu")]
HEADERS = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + \
    [os.path.join(ROOT, "include", "topk_packed.h")]
OUTPUT = os.path.join(PKG, "libtopk_packed.so")
OUTPUT_CHECKED = os.path.join(PKG, "libtopk_packed_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def command(output: str = OUTPUT, ptxas_verbose: bool = False, checked: bool = False) -> list[str]:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-Xlinker", "-Bsymbolic", "-I", os.path.join(ROOT, "include"),
           "-o", output, *SOURCES]
    if checked:
        cmd.insert(1, "-DTOPK_CHECKED")
    if ptxas_verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def up_to_date(output: str = OUTPUT) -> bool:
    if not os.path.exists(output):
        return False
    t = os.path.getmtime(output)
    return all(os.path.getmtime(f) <= t for f in SOURCES + HEADERS)


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    """Builds both libraries (those not up to date); returns the normal one's path."""
    jobs = [(out, checked) for out, checked in ((OUTPUT, False), (OUTPUT_CHECKED, True))
            if force or ptxas_verbose or not up_to_date(out)]
    procs = [(subprocess.Popen(command(out, ptxas_verbose, checked)), out) for out, checked in jobs]
    failed = [out for proc, out in procs if proc.wait() != 0]
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(os.path.basename(f) for f in failed))
    return OUTPUT


if __name__ == "__main__":
    print(build(force=True, ptxas_verbose="--verbose-ptxas" in sys.argv))
