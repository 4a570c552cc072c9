"""Builds the CPU oracle in-tree: oracle/libmoe_oracle.so (gcc, C11, fp64, OpenMP).

TEST INFRASTRUCTURE ONLY.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libmoe_oracle.so")
SRC = [os.path.join(HERE, "moe_oracle.c")]
HDR = [os.path.join(HERE, "moe_oracle.h")]


def build(force=False):
    stale = not os.path.exists(LIB) or any(os.path.getmtime(s) > os.path.getmtime(LIB) for s in SRC + HDR)
    if force or stale:
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
               "-o", LIB] + SRC + ["-lm"]
        subprocess.check_call(cmd)
    return LIB


if __name__ == "__main__":
    build(force=True)
