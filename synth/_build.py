"""Compile the seeded input generators: host (C) and device (CUDA, sm_103a)."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def commands(nvcc="nvcc"):
    host = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
            "-Wall", "-o", os.path.join(HERE, "libsynth_host.so"),
            os.path.join(HERE, "synth_host.c")]
    dev = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
           "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-fmad=false",
           "-o", os.path.join(HERE, "libsynth_dev.so"), os.path.join(HERE, "synth_dev.cu")]
    return [host, dev]
