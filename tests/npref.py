"""An independent numpy derivation of the layer, used only to pin the C oracle.

It shares no code with the oracle: element values come from the hand-typed OCP
table in tests/golden, unpacking uses numpy bit operations, matrix products use
numpy's matmul, top-k uses a full lexicographic sort and the gates use the full
softmax over all E experts, restricted to the selected ones and renormalised.
"""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

with open(os.path.join(GOLDEN, "e2m1_ocp_mx.json")) as _f:
    E2M1_TABLE = np.array(json.load(_f)["values"], dtype=np.float64)


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def f16_to_f64(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def to_f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_to_f64(a)
    return a.astype(np.float64)


def unpack_mxfp4(codes, scales, rows, K):
    codes = np.asarray(codes, dtype=np.uint8).reshape(rows, K // 2)
    scales = np.asarray(scales, dtype=np.uint8).reshape(rows, K // 32)
    nib = np.empty((rows, K), dtype=np.uint8)
    nib[:, 0::2] = codes & 0x0F
    nib[:, 1::2] = codes >> 4
    vals = E2M1_TABLE[nib]
    sc = np.where(scales == 255, np.nan, np.exp2(scales.astype(np.float64) - 127.0))
    return vals * np.repeat(sc, 32, axis=1)


def unpack_rvq3(codes, cb, rows, K):
    codes = np.asarray(codes, dtype=np.uint8).reshape(3, K // 8, rows).transpose(0, 2, 1)  # -> [s][r][v]
    cbf = f16_to_f64(np.asarray(cb).reshape(3, 256, 8))
    w = cbf[0][codes[0]] + cbf[1][codes[1]] + cbf[2][codes[2]]  # [rows][K/8][8]
    return w.reshape(rows, K)


def mxfp4_record_mats(rec, d, ff):
    rec = np.asarray(rec, dtype=np.uint8)
    cb, sb = ff * d // 2, ff * d // 32
    o = 0
    mats = []
    for rows, K in ((ff, d), (ff, d), (d, ff)):
        codes = rec[o:o + rows * K // 2]
        o += rows * K // 2
        scales = rec[o:o + rows * K // 32]
        o += rows * K // 32
        mats.append(unpack_mxfp4(codes, scales, rows, K))
    assert o == 3 * (cb + sb)
    return mats


def rvq3_record_mats(rec, cbs, d, ff):
    rec = np.asarray(rec, dtype=np.uint8)
    mb = 3 * ff * d // 8
    return [unpack_rvq3(rec[0:mb], cbs[0], ff, d), unpack_rvq3(rec[mb:2 * mb], cbs[1], ff, d),
            unpack_rvq3(rec[2 * mb:3 * mb], cbs[2], d, ff)]


def silu(g):
    return g / (1.0 + np.exp(-g))


def expert(x, mats, act="swiglu"):
    wg, wu, wd = mats
    g = wg @ x
    u = wu @ x
    if act == "swiglu":
        h = silu(g) * u
    else:
        sig = 1.0 / (1.0 + np.exp(-g))
        h = 4.0 * np.tanh(g / 4.0) * sig * 25.0 * np.tanh(u / 25.0)
    return wd @ h


def topk_sorted(logits, k):
    """Full sort per token by (logit descending, expert ascending)."""
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))
        idx[t] = order[:k]
    return idx


def gates_full_softmax(logits, idx):
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, idx, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def layer(x, W, bias, k, expert_mats, act="swiglu", bias_mode="logit", n_shared=0):
    """bias_mode "select": the bias only chooses the experts, the gates come from
    the logits without it.  Experts E .. E + n_shared - 1 are shared: every
    token adds their outputs unweighted."""
    xf = to_f64(x)
    plain = xf @ to_f64(W).T
    logits = plain
    if bias is not None:
        logits = plain + np.asarray(bias, dtype=np.float64)[None, :]
    idx = topk_sorted(logits, k)
    g = gates_full_softmax(plain if bias_mode == "select" else logits, idx)
    T, d = xf.shape
    E = W.shape[0]
    delta = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            if g[t, j] != 0.0:
                delta[t] += g[t, j] * expert(xf[t], expert_mats(int(idx[t, j])), act)
        for s in range(n_shared):
            delta[t] += expert(xf[t], expert_mats(E + s), act)
    return logits, idx, g, delta


def fnv1a64(arr):
    """FNV-1a (64-bit) over the bytes of an array: equal hash <=> equal bytes (w.h.p.)."""
    h = 0xCBF29CE484222325
    for b in np.ascontiguousarray(arr).view(np.uint8).tobytes():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h
