"""Build recipe of libsv.so (sm_103a): one nvcc compile per translation unit,
run in parallel by the caller, then one link."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsv.so")
SOURCES = ["k_linear.cu", "k_linear_tc.cu", "k_attn.cu", "k_misc.cu", "sv_api.cu", "sv_noalloc.cu"]

# --fmad=false: every fused multiply-add in the kernels is written out, so
# the rounding of each element never depends on what the compiler contracts.
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--fmad=false", "-Xcompiler", "-fPIC",
         "-I", os.path.join(HERE, "..", "include")]


def jobs(nvcc: str, arch: list[str]):
    os.makedirs(OBJ, exist_ok=True)
    out = []
    for src in SOURCES:
        obj = os.path.join(OBJ, src.replace(".cu", ".o"))
        out.append(([nvcc, *arch, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj], f"csrc/{src}"))
    return out


def link(nvcc: str, arch: list[str]) -> None:
    objs = [os.path.join(OBJ, s.replace(".cu", ".o")) for s in SOURCES]
    tmp = LIB + ".tmp"
    subprocess.run([nvcc, *arch, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
