"""ctypes wrapper of the fp64 CPU oracle (oracle/moe_oracle.c).

TEST INFRASTRUCTURE ONLY.  Imported by tests/, by __graft_entry__.smoke() and
by bench.py's CPU-baseline leg; the product path never imports it.

Arrays: x and router W are numpy float32 (fp32) or uint16 (bfloat16 bit
patterns); records are uint8 arrays; codebooks are uint16 fp16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
ACT = {"swiglu": 0, "situ": 1}
QUANT = {"mxfp4": 0, "rvq3": 1}

_lib = None


def lib():
    global _lib
    if _lib is None:
        # MOE_ORACLE_LIB points the tests' mutation check at a deliberately broken copy
        L = ctypes.CDLL(os.environ.get("MOE_ORACLE_LIB") or _build.build())
        vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.or_e2m1.argtypes, L.or_e2m1.restype = [i32], dbl
        L.or_e8m0.argtypes, L.or_e8m0.restype = [i32], dbl
        L.or_bf16.argtypes, L.or_bf16.restype = [ctypes.c_uint16], dbl
        L.or_f16.argtypes, L.or_f16.restype = [ctypes.c_uint16], dbl
        L.or_act.argtypes, L.or_act.restype = [dbl, dbl, i32], dbl
        L.or_mxfp4_row.argtypes = [vp, vp, i32, i32, vp]
        L.or_rvq3_row.argtypes = [vp, vp, i32, i32, i32, vp]
        L.or_rvq3_row_rowmajor.argtypes = [vp, vp, i32, i32, i32, vp]
        L.or_mxfp4_record_bytes.argtypes, L.or_mxfp4_record_bytes.restype = [i32, i32], ctypes.c_size_t
        L.or_rvq3_record_bytes.argtypes, L.or_rvq3_record_bytes.restype = [i32, i32], ctypes.c_size_t
        L.or_router.argtypes = [vp, i32, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp]
        L.or_crc32.argtypes, L.or_crc32.restype = [vp, ctypes.c_size_t], ctypes.c_uint32
        L.or_router_mode.argtypes = [vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, vp, vp, vp]
        L.or_topk_gates.argtypes = [vp, i32, i32, i32, vp, vp]
        L.or_bucket.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.or_expert_mxfp4.argtypes = [vp, vp, i32, i32, i32, vp]
        L.or_expert_rvq3.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp]
        L.or_expert_rvq3_rowmajor.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp]
        L.or_combine.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.or_layer_forward.argtypes = [vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                       vp, i32, vp, vp, vp, vp]
        L.or_layer_forward_ex.argtypes = [vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp,
                                          vp, vp, vp, i32, vp, vp, vp, vp]
        L.or_partial_delta.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, i32, i32,
                                       vp]
        L.or_project.argtypes = [vp, i32, vp, i32, i32, i32, i32, vp]
        L.or_round_bf16.argtypes, L.or_round_bf16.restype = [ctypes.c_double], ctypes.c_uint16
        L.or_latent_forward.argtypes = [vp, i32, vp, vp, i32, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                        i32, i32, vp, vp, vp, vp, i32, vp, vp]
        for f in ("or_router", "or_topk_gates", "or_bucket", "or_expert_mxfp4", "or_expert_rvq3",
                  "or_expert_rvq3_rowmajor", "or_combine",
                  "or_layer_forward", "or_partial_delta", "or_project", "or_latent_forward"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _dt(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"unsupported dtype {a.dtype}")


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} returned {rc}")


def e2m1(code):
    return lib().or_e2m1(int(code))


def e8m0(byte):
    return lib().or_e8m0(int(byte))


def bf16(bits):
    return lib().or_bf16(int(bits))


def f16(bits):
    return lib().or_f16(int(bits))


def act(g, u, kind="swiglu"):
    return lib().or_act(float(g), float(u), ACT[kind])


def mxfp4_row(codes, scales, K, r):
    w = np.empty(K, dtype=np.float64)
    lib().or_mxfp4_row(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(scales)), K, r, _p(w))
    return w


def mxfp4_matrix(codes, scales, rows, K):
    return np.stack([mxfp4_row(codes, scales, K, r) for r in range(rows)])


def rvq3_row(codes, cb, rows, K, r):
    w = np.empty(K, dtype=np.float64)
    lib().or_rvq3_row(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(cb)), rows, K, r, _p(w))
    return w


def rvq3_matrix(codes, cb, rows, K):
    return np.stack([rvq3_row(codes, cb, rows, K, r) for r in range(rows)])


def rvq3_row_rowmajor(codes, cb, rows, K, r):
    w = np.empty(K, dtype=np.float64)
    lib().or_rvq3_row_rowmajor(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(cb)), rows, K, r, _p(w))
    return w


def rvq3_matrix_rowmajor(codes, cb, rows, K):
    return np.stack([rvq3_row_rowmajor(codes, cb, rows, K, r) for r in range(rows)])


def mxfp4_record_bytes(d, ff):
    return int(lib().or_mxfp4_record_bytes(d, ff))


def rvq3_record_bytes(d, ff):
    return int(lib().or_rvq3_record_bytes(d, ff))


def crc32(data):
    """CRC-32 (IEEE, as zlib) of a byte string or uint8 array."""
    a = np.frombuffer(bytes(data), dtype=np.uint8) if isinstance(data, (bytes, bytearray)) else \
        np.ascontiguousarray(data, dtype=np.uint8).reshape(-1)
    return int(lib().or_crc32(_p(a) if a.size else None, a.size))


BIAS_MODE = {"logit": 0, "select": 1}


def router(x, W, bias, k, bias_mode="logit"):
    """Returns (selection keys l + bias [T][E], topk_idx [T][k], gates [T][k]).
    bias_mode "logit": the bias enters selection and gates; "select": the
    selection only (gates from the logits without it)."""
    x = np.ascontiguousarray(x)
    W = np.ascontiguousarray(W)
    T, d = x.shape
    E = W.shape[0]
    logits = np.empty((T, E), dtype=np.float64)
    idx = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _check(lib().or_router_mode(_p(x), _dt(x), _p(W), _dt(W), _p(b), BIAS_MODE[bias_mode], T, d, E, k, _p(logits),
                                _p(idx), _p(gates)), "router")
    return logits, idx, gates


def topk_gates(logits, k):
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    _check(lib().or_topk_gates(_p(logits), T, E, k, _p(idx), _p(gates)), "topk_gates")
    return idx, gates


def bucket(topk_idx, E):
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = topk_idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    pair_ids = np.empty(T * k, dtype=np.int32)
    _check(lib().or_bucket(_p(topk_idx), T, k, E, _p(counts), _p(offsets), _p(pair_ids)), "bucket")
    return counts, offsets, pair_ids


def expert_mxfp4(x, rec, d, ff, act_kind="swiglu"):
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(d, dtype=np.float64)
    _check(lib().or_expert_mxfp4(_p(x), _p(np.ascontiguousarray(rec)), d, ff, ACT[act_kind], _p(y)), "expert_mxfp4")
    return y


def expert_rvq3(x, rec, cb_gate, cb_up, cb_down, d, ff, act_kind="swiglu"):
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(d, dtype=np.float64)
    _check(lib().or_expert_rvq3(_p(x), _p(np.ascontiguousarray(rec)), _p(cb_gate), _p(cb_up), _p(cb_down), d, ff,
                                ACT[act_kind], _p(y)), "expert_rvq3")
    return y


def expert_rvq3_rowmajor(x, rec, cb_gate, cb_up, cb_down, d, ff, act_kind="swiglu"):
    """expert_rvq3 on a record whose code planes are stored row by row."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(d, dtype=np.float64)
    _check(lib().or_expert_rvq3_rowmajor(_p(x), _p(np.ascontiguousarray(rec)), _p(cb_gate), _p(cb_up), _p(cb_down),
                                         d, ff, ACT[act_kind], _p(y)), "expert_rvq3_rowmajor")
    return y


def combine(x_resid, y_pairs, gates, k):
    y_pairs = np.ascontiguousarray(y_pairs, dtype=np.float64)
    gates = np.ascontiguousarray(gates, dtype=np.float64)
    P, d = y_pairs.shape
    T = P // k
    out = np.empty((T, d), dtype=np.float64)
    xr = None if x_resid is None else np.ascontiguousarray(x_resid, dtype=np.float64)
    _check(lib().or_combine(_p(xr), _p(y_pairs), _p(gates), T, k, d, _p(out)), "combine")
    return out


def _records_array(records, E):
    arr = (ctypes.c_void_p * E)()
    keep = []
    for e in range(E):
        r = records.get(e) if isinstance(records, dict) else records[e]
        if r is not None:
            r = np.ascontiguousarray(r, dtype=np.uint8)
            keep.append(r)
            arr[e] = r.ctypes.data
        else:
            arr[e] = None
    return arr, keep


def layer_forward(x, W, bias, d, ff, E, k, records, quant="mxfp4", act_kind="swiglu", codebooks=None,
                  token_mask=None, nthreads=1, n_shared=0, bias_mode="logit"):
    """Returns (topk_idx [T][k], gates [T][k], y_delta [T][d], out [T][d]) in fp64.
    records: list/dict expert -> uint8 record (None = absent), E + n_shared
    entries: records[E + s] is shared expert s (every token, weight 1).
    codebooks: (cb_gate, cb_up, cb_down) fp16 [3][256][8] arrays for RVQ3.
    Rows of tokens outside token_mask come back as NaN."""
    x = np.ascontiguousarray(x)
    W = np.ascontiguousarray(W)
    T = x.shape[0]
    idx = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    y = np.full((T, d), np.nan)
    out = np.full((T, d), np.nan)
    arr, keep = _records_array(records, E + n_shared)
    cbs = [None, None, None] if codebooks is None else [np.ascontiguousarray(c, dtype=np.uint16) for c in codebooks]
    mask = None if token_mask is None else np.ascontiguousarray(token_mask, dtype=np.uint8)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rc = lib().or_layer_forward_ex(_p(x), _dt(x), _p(W), _dt(W), _p(b), BIAS_MODE[bias_mode], T, d, ff, E, k,
                                   int(n_shared), ACT[act_kind], QUANT[quant], ctypes.cast(arr, ctypes.c_void_p),
                                   _p(cbs[0]), _p(cbs[1]), _p(cbs[2]), _p(mask), int(nthreads), _p(idx), _p(gates),
                                   _p(y), _p(out))
    del keep
    _check(rc, "layer_forward")
    return idx, gates, y, out


def partial_delta(x, topk_idx, gates, d, ff, k, records, e_begin, e_end, quant="mxfp4", act_kind="swiglu",
                  codebooks=None):
    x = np.ascontiguousarray(x)
    T = x.shape[0]
    E = max(e_end, int(topk_idx.max()) + 1)
    arr, keep = _records_array(records, E) if isinstance(records, dict) else _records_array(list(records), E)
    cbs = [None, None, None] if codebooks is None else [np.ascontiguousarray(c, dtype=np.uint16) for c in codebooks]
    delta = np.empty((T, d), dtype=np.float64)
    rc = lib().or_partial_delta(_p(x), _dt(x), _p(np.ascontiguousarray(topk_idx, dtype=np.int32)),
                                _p(np.ascontiguousarray(gates, dtype=np.float64)), T, d, ff, k, ACT[act_kind],
                                QUANT[quant], ctypes.cast(arr, ctypes.c_void_p), _p(cbs[0]), _p(cbs[1]),
                                _p(cbs[2]), e_begin, e_end, _p(delta))
    del keep
    _check(rc, "partial_delta")
    return delta


def project(x, W):
    """y[t][n] = sum_k W[n][k] x[t][k] in fp64 (x [T][K], W [N][K]; float32 or
    bf16 bit patterns in uint16)."""
    x = np.ascontiguousarray(x)
    W = np.ascontiguousarray(W)
    T, K = x.shape
    N = W.shape[0]
    y = np.empty((T, N), dtype=np.float64)
    _check(lib().or_project(_p(x), _dt(x), _p(W), _dt(W), T, K, N, _p(y)), "project")
    return y


def round_bf16(v):
    """bf16 bit patterns (uint16) of the values in v, rounded to nearest even."""
    a = np.asarray(v, dtype=np.float64)
    f = lib().or_round_bf16
    return np.array([f(float(t)) for t in a.reshape(-1)], dtype=np.uint16).reshape(a.shape)


def latent_forward(x, w_in, w_out, router_w, bias, d, ff, E, k, records, quant="mxfp4", act_kind="swiglu",
                   codebooks=None, nthreads=1, n_shared=0, bias_mode="logit"):
    """(z bf16 bits [T][d], out [T][D]) of the layer run in the latent space:
    z = bf16(W_in x), out = x + W_out (MoE delta of z)."""
    x = np.ascontiguousarray(x)
    w_in = np.ascontiguousarray(w_in)
    w_out = np.ascontiguousarray(w_out)
    assert _dt(w_in) == _dt(w_out)
    T, D = x.shape
    z = np.empty((T, d), dtype=np.uint16)
    out = np.empty((T, D), dtype=np.float64)
    recs, keep = _records_array(records, E + n_shared)
    cbs = codebooks if codebooks is not None else (None, None, None)
    rw = np.ascontiguousarray(router_w)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _check(lib().or_latent_forward(_p(x), _dt(x), _p(w_in), _p(w_out), _dt(w_in), D, _p(rw), _dt(rw), _p(b),
                                   BIAS_MODE[bias_mode], T, d, ff, E, k, n_shared, ACT[act_kind], QUANT[quant], recs,
                                   _p(cbs[0]), _p(cbs[1]), _p(cbs[2]), int(nthreads), _p(z), _p(out)),
           "latent_forward")
    return z, out
