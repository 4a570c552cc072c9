"""Builds the CPU oracle in-tree: oracle/libmoe_oracle.so (gcc, C11, fp64, OpenMP).

TEST INFRASTRUCTURE ONLY.
"""
import fcntl
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libmoe_oracle.so")
SRC = [os.path.join(HERE, "moe_oracle.c")]
HDR = [os.path.join(HERE, "moe_oracle.h")]


def _stale():
    return not os.path.exists(LIB) or any(os.path.getmtime(s) > os.path.getmtime(LIB) for s in SRC + HDR)


def build(force=False):
    if not (force or _stale()):
        return LIB
    with open(os.path.join(HERE, ".build.lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)  # one builder at a time; others reuse its result
        if force or _stale():
            tmp = LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
                   "-o", tmp] + SRC + ["-lm"]
            subprocess.check_call(cmd)
            os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True)
