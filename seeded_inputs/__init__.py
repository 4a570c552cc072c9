"""Seeded synthetic inputs for the MoE-layer forward.

This module is the only code shared by the CPU oracle's drivers and the GPU
path's drivers.  It turns (seed, stream, index) into bytes and holds none of
the layer's arithmetic.  Host fills return numpy arrays; device fills write
into caller-owned device memory given as raw pointers (no torch import here).
"""
import ctypes
import os

import numpy as np

from . import build as _build
from .workloads import LayerRecipe, WORKLOADS, get_workload  # noqa: F401

STREAM_X = 1
STREAM_ROUTER_W = 2
STREAM_CODEBOOK = 16
STREAM_RECORD = 0x100000

_DT = {"f32": 0, "bf16": 1, "f16": 2}
_NP = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16}

_host = None
_cuda = None


def host_lib():
    global _host
    if _host is None:
        path = _build.build_host()
        lib = ctypes.CDLL(path)
        u64, i32, vp, dbl = ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        lib.si_fill_normal.argtypes = [u64, u64, dbl, u64, u64, i32, vp]
        lib.si_fill_bytes.argtypes = [u64, u64, u64, u64, vp]
        lib.si_mxfp4_record_size.argtypes = [u64, u64]
        lib.si_mxfp4_record_size.restype = u64
        lib.si_rvq3_record_size.argtypes = [u64, u64]
        lib.si_rvq3_record_size.restype = u64
        lib.si_fill_mxfp4_record.argtypes = [u64, u64, u64, u64, ctypes.c_uint32, ctypes.c_uint32, u64, u64, vp]
        lib.si_fill_rvq3_record.argtypes = [u64, u64, u64, u64, vp]
        _host = lib
    return _host


def cuda_lib():
    """The device filler; raises if it cannot be built or loaded."""
    global _cuda
    if _cuda is None:
        path = _build.build_cuda()
        if path is None:
            raise RuntimeError("seeded_inputs: nvcc not found, cannot build the device filler")
        lib = ctypes.CDLL(path)
        u64, i32, vp, dbl = ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        lib.si_dev_fill_normal.argtypes = [u64, u64, dbl, u64, u64, i32, vp, vp]
        lib.si_dev_fill_bytes.argtypes = [u64, u64, u64, u64, vp, vp]
        lib.si_dev_fill_mxfp4_bank.argtypes = [u64, u64, u64, u64, u64, ctypes.c_uint32, ctypes.c_uint32, vp,
                                               u64, vp]
        lib.si_dev_fill_rvq3_bank.argtypes = [u64, u64, u64, u64, u64, vp, u64, vp]
        for f in (lib.si_dev_fill_normal, lib.si_dev_fill_bytes, lib.si_dev_fill_mxfp4_bank,
                  lib.si_dev_fill_rvq3_bank):
            f.restype = i32
        _cuda = lib
    return _cuda


# ----------------------------------------------------------------------------- host fills

def normal(seed, stream, sigma, n, dtype="f32", offset=0):
    """n variates of N(0, sigma^2) (Irwin-Hall(12) shape), stored as f32, or as
    bf16 / f16 bit patterns in uint16."""
    out = np.empty(n, dtype=_NP[dtype])
    host_lib().si_fill_normal(seed, stream, float(sigma), offset, n, _DT[dtype], out.ctypes.data)
    return out


def uniform_bytes(seed, stream, n, offset=0):
    out = np.empty(n, dtype=np.uint8)
    host_lib().si_fill_bytes(seed, stream, offset, n, out.ctypes.data)
    return out


def mxfp4_record_size(d, ff):
    return int(host_lib().si_mxfp4_record_size(d, ff))


def rvq3_record_size(d, ff):
    return int(host_lib().si_rvq3_record_size(d, ff))


def mxfp4_record(seed, expert, d, ff, scale_lo, scale_hi, offset=0, n=None):
    if n is None:
        n = mxfp4_record_size(d, ff) - offset
    out = np.empty(n, dtype=np.uint8)
    host_lib().si_fill_mxfp4_record(seed, expert, d, ff, scale_lo, scale_hi, offset, n, out.ctypes.data)
    return out


def rvq3_record(seed, expert, d, ff, offset=0, n=None):
    if n is None:
        n = rvq3_record_size(d, ff) - offset
    out = np.empty(n, dtype=np.uint8)
    host_lib().si_fill_rvq3_record(seed, expert, offset, n, out.ctypes.data)
    return out


def zipf_bias(E, s=1.0):
    """Additive router-logit bias b[e] = -s * ln(e + 1): the log of a Zipf(s)
    prior over expert ids with rank = id + 1 (computed once, on the host)."""
    return (-s * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


# ----------------------------------------------------------------------------- layer inputs (host)

def layer_x(r: "LayerRecipe", T=None, token_offset=0):
    T = r.T if T is None else T
    return normal(r.seed, STREAM_X, r.x_sigma, T * r.d, r.x_dtype, offset=token_offset * r.d).reshape(T, r.d)


def layer_router_w(r: "LayerRecipe"):
    return normal(r.seed, STREAM_ROUTER_W, r.w_sigma, r.E * r.d, r.w_dtype).reshape(r.E, r.d)


def layer_bias(r: "LayerRecipe"):
    if r.bias == "zipf":
        return zipf_bias(r.E, r.zipf_s)
    return None


def layer_codebooks(r: "LayerRecipe"):
    """fp16 bit patterns [3][256][8]; stage s (0-based) has std 0.02 / (s + 1)."""
    cb = np.empty((3, 256, 8), dtype=np.uint16)
    for s in range(3):
        cb[s] = normal(r.seed, STREAM_CODEBOOK + s, 0.02 / (s + 1), 256 * 8, "f16").reshape(256, 8)
    return cb


def layer_record(r: "LayerRecipe", expert):
    if r.quant == "mxfp4":
        return mxfp4_record(r.seed, expert, r.d, r.ff, r.scale_lo, r.scale_hi)
    return rvq3_record(r.seed, expert, r.d, r.ff)


def layer_records(r: "LayerRecipe", experts, n_total=None, nthreads=None):
    """A list of n_total (default E + n_shared) entries: the record of each
    expert in `experts`, None elsewhere; the records are generated on
    `nthreads` host threads (the C filler runs without the GIL)."""
    import concurrent.futures as cf
    n_total = r.E + r.n_shared if n_total is None else n_total
    want = sorted(set(int(e) for e in experts))
    out = [None] * n_total
    nthreads = nthreads or min(32, os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=max(1, nthreads)) as ex:
        for e, rec in zip(want, ex.map(lambda e: layer_record(r, e), want)):
            out[e] = rec
    return out


def record_size(r: "LayerRecipe"):
    return mxfp4_record_size(r.d, r.ff) if r.quant == "mxfp4" else rvq3_record_size(r.d, r.ff)


# ----------------------------------------------------------------------------- device fills

def _chk(rc, what):
    if rc != 0:
        raise RuntimeError(f"seeded_inputs: {what} failed (code {rc})")


def dev_normal(ptr, seed, stream, sigma, n, dtype="f32", offset=0, cuda_stream=0):
    _chk(cuda_lib().si_dev_fill_normal(seed, stream, float(sigma), offset, n, _DT[dtype], ptr, cuda_stream),
         "si_dev_fill_normal")


def dev_uniform_bytes(ptr, seed, stream, n, offset=0, cuda_stream=0):
    _chk(cuda_lib().si_dev_fill_bytes(seed, stream, offset, n, ptr, cuda_stream), "si_dev_fill_bytes")


def dev_record_bank(r: "LayerRecipe", ptr, stride, e0=0, n_exp=None, cuda_stream=0):
    n_exp = r.E - e0 if n_exp is None else n_exp
    if r.quant == "mxfp4":
        rc = cuda_lib().si_dev_fill_mxfp4_bank(r.seed, e0, n_exp, r.d, r.ff, r.scale_lo, r.scale_hi, ptr, stride,
                                               cuda_stream)
    else:
        rc = cuda_lib().si_dev_fill_rvq3_bank(r.seed, e0, n_exp, r.d, r.ff, ptr, stride, cuda_stream)
    _chk(rc, "device record bank fill")


def dev_layer_x(r: "LayerRecipe", ptr, T=None, token_offset=0, cuda_stream=0):
    T = r.T if T is None else T
    dev_normal(ptr, r.seed, STREAM_X, r.x_sigma, T * r.d, r.x_dtype, offset=token_offset * r.d,
               cuda_stream=cuda_stream)


def dev_layer_router_w(r: "LayerRecipe", ptr, cuda_stream=0):
    dev_normal(ptr, r.seed, STREAM_ROUTER_W, r.w_sigma, r.E * r.d, r.w_dtype, cuda_stream=cuda_stream)


def dev_layer_codebooks(r: "LayerRecipe", ptr, cuda_stream=0):
    for s in range(3):
        dev_normal(ptr + s * 256 * 8 * 2, r.seed, STREAM_CODEBOOK + s, 0.02 / (s + 1), 256 * 8, "f16",
                   cuda_stream=cuda_stream)
