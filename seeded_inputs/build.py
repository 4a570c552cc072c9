"""Builds the seeded-input generator libraries in-tree.

libseeded_inputs_host.so  -- gcc, always built (the CPU tests need it).
libseeded_inputs_cuda.so  -- nvcc for sm_103a, built when nvcc is present.
"""
import fcntl
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libseeded_inputs_host.so")
CUDA_LIB = os.path.join(HERE, "libseeded_inputs_cuda.so")
_HOST_SRC = [os.path.join(HERE, "si_host.c")]
_CUDA_SRC = [os.path.join(HERE, "si_device.cu")]
_HDR = [os.path.join(HERE, "si_rng.h")]


def _stale(out, srcs):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand if os.path.exists(cand) else None


def _locked_build(out, srcs, make_cmd, force):
    if not (force or _stale(out, srcs)):
        return out
    with open(os.path.join(HERE, ".build.lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)  # one builder at a time; others reuse its result
        if force or _stale(out, srcs):
            tmp = out + f".tmp{os.getpid()}"
            subprocess.check_call(make_cmd(tmp))
            os.replace(tmp, out)
    return out


def build_host(force=False):
    return _locked_build(HOST_LIB, _HOST_SRC + _HDR, lambda o: ["gcc", "-O2", "-std=c11", "-ffp-contract=off",
                                                                 "-fPIC", "-shared", "-o", o] + _HOST_SRC, force)


def build_cuda(force=False):
    nvcc = _nvcc()
    if nvcc is None:
        return None
    return _locked_build(CUDA_LIB, _CUDA_SRC + _HDR,
                         lambda o: [nvcc, "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                                    "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC", "-shared", "-o", o]
                         + _CUDA_SRC, force)


def build(force=False):
    build_host(force)
    build_cuda(force)


if __name__ == "__main__":
    build(force=True)
