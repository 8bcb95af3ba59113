"""Compile the CUDA library (sm_103a) in-tree: one object per kernel file,
compiled in parallel, linked into libmoe_decode.so next to this file."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_decode.so")
# the bounds-check variant (MOE_BOUNDS_CHECK): data-dependent indexes tested
# before use, latching an error instead of faulting; loaded by the binding
# when MOE_DECODE_LIB names it
BUILD_BOUNDS = os.path.join(HERE, "_build_bounds")
LIB_BOUNDS = os.path.join(HERE, "libmoe_decode_bounds.so")
SOURCES = ["boundary.cu", "router.cu", "experts.cu", "experts_tc.cu", "tc_gemm.cu", "quant.cu", "quant_noalloc.cu",
           "dense.cu", "ctxkv.cu", "capi.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr"]


def compile_commands(nvcc="nvcc", extra=(), build_dir=BUILD):
    """[(object path, argv)] for every source."""
    out = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        out.append((obj, [nvcc, *ARCH, *FLAGS, *extra, "-I", CSRC, "-c",
                          os.path.join(CSRC, src), "-o", obj]))
    return out


def link_command(objects, nvcc="nvcc", lib=LIB):
    return [nvcc, *ARCH, "-shared", "-o", lib, *objects]
