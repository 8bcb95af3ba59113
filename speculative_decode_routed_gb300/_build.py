"""Compile the CUDA library (sm_103a) in-tree: one object per kernel file,
compiled in parallel, linked into libmoe_decode.so next to this file."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_decode.so")
SOURCES = ["boundary.cu", "router.cu", "experts.cu", "experts_tc.cu", "quant.cu", "quant_noalloc.cu", "dense.cu", "ctxkv.cu", "capi.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr"]


def compile_commands(nvcc="nvcc", extra=()):
    """[(object path, argv)] for every source."""
    out = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        out.append((obj, [nvcc, *ARCH, *FLAGS, *extra, "-I", CSRC, "-c",
                          os.path.join(CSRC, src), "-o", obj]))
    return out


def link_command(objects, nvcc="nvcc"):
    return [nvcc, *ARCH, "-shared", "-o", LIB, *objects, "-lcublas"]
