"""Compile the CPU oracle (plain C, OpenMP) into oracle/liboracle.so."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def commands():
    src = os.path.join(HERE, "oracle.c")
    out = os.path.join(HERE, "liboracle.so")
    # -ffp-contract=off: every fp32 operation the definitions spell out is
    # rounded on its own, never fused into a multiply-add.
    return [["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
             "-Wall", "-Wextra", "-o", out, src, "-lm"]]
