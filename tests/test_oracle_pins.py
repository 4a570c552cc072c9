"""Pins the CPU oracle to facts that do not come from the oracle itself.

Each test names the mistake it is meant to catch.  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import npref

GOLDEN = npref.GOLDEN


# ----------------------------------------------------------------------------- element decodes

def test_e2m1_all_codes_match_ocp_table():
    # catches a wrong exponent bias, a swapped sign bit or a wrong subnormal rule
    for c in range(16):
        v = oracle.e2m1(c)
        assert v == npref.E2M1_TABLE[c]
        assert math.copysign(1.0, v) == math.copysign(1.0, npref.E2M1_TABLE[c])  # -0.0 for code 8


def test_e8m0_all_bytes_and_products():
    # all 16 codes x 256 scale bytes against 2^(b-127) from math.ldexp
    for b in range(256):
        s = oracle.e8m0(b)
        if b == 255:
            assert math.isnan(s)
            continue
        assert s == math.ldexp(1.0, b - 127)
        for c in range(16):
            codes = np.full(1, c | (c << 4), dtype=np.uint8)
            w = oracle.mxfp4_row(np.tile(codes, 16), np.full(1, b, dtype=np.uint8), 32, 0)
            assert np.all(w == npref.E2M1_TABLE[c] * math.ldexp(1.0, b - 127))


def test_bf16_f16_decodes_match_numpy():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    for b in bits:
        f = npref.f16_to_f64(np.array([b]))[0]
        o = oracle.f16(int(b))
        assert (np.isnan(f) and np.isnan(o)) or f == o
    for b in bits[::5]:
        f = npref.bf16_to_f64(np.array([b]))[0]
        o = oracle.bf16(int(b))
        assert (np.isnan(f) and np.isnan(o)) or f == o


def test_mxfp4_row_nibble_order_and_block_scales():
    # catches low/high nibble swaps and a scale block applied to the wrong columns
    rng = np.random.default_rng(7)
    rows, K = 5, 128
    codes = rng.integers(0, 256, size=rows * K // 2, dtype=np.uint8)
    scales = rng.integers(100, 140, size=rows * K // 32, dtype=np.uint8)
    ref = npref.unpack_mxfp4(codes, scales, rows, K)
    got = oracle.mxfp4_matrix(codes, scales, rows, K)
    np.testing.assert_array_equal(got, ref)
    # column 0 is the low nibble of byte 0
    codes2 = np.zeros(K // 2, dtype=np.uint8)
    codes2[0] = 0x72  # col0 = code 2 (1.0), col1 = code 7 (6.0)
    w = oracle.mxfp4_row(codes2, np.full(K // 32, 127, dtype=np.uint8), K, 0)
    assert w[0] == 1.0 and w[1] == 6.0 and np.all(w[2:] == 0.0)


def test_rvq3_is_sum_of_three_codewords():
    rng = np.random.default_rng(3)
    rows, K = 6, 64
    codes = rng.integers(0, 256, size=3 * rows * K // 8, dtype=np.uint8)
    cb = si.normal(11, 16, 0.02, 3 * 256 * 8, "f16").reshape(3, 256, 8)
    got = oracle.rvq3_matrix(codes, cb, rows, K)
    np.testing.assert_array_equal(got, npref.unpack_rvq3(codes, cb, rows, K))
    # stages 2 and 3 zeroed: a plain vector-quantisation table lookup
    cb0 = cb.copy()
    cb0[1:] = 0
    got0 = oracle.rvq3_matrix(codes, cb0, rows, K)
    c0 = codes.reshape(3, K // 8, rows)[0].T  # code[0][v][r] -> [r][v]
    for r in range(rows):
        for v in range(K // 8):
            for i in range(8):
                assert got0[r, 8 * v + i] == npref.f16_to_f64(np.array([cb[0, c0[r, v], i]]))[0]


def test_rvq3_row_major_reader_is_the_same_definition():
    # codes stored row by row, [3][rows][K/8]: every weight is the sum of the
    # three stages' codeword components, written out here index by index
    rng = np.random.default_rng(5)
    rows, K = 5, 48
    nv = K // 8
    codes = rng.integers(0, 256, size=3 * rows * nv, dtype=np.uint8)
    cb = si.normal(12, 16, 0.02, 3 * 256 * 8, "f16").reshape(3, 256, 8)
    cbf = npref.f16_to_f64(cb.reshape(-1)).reshape(3, 256, 8)
    got = oracle.rvq3_matrix_rowmajor(codes, cb, rows, K)
    for r in range(rows):
        for v in range(nv):
            for i in range(8):
                want = 0.0
                for s in range(3):
                    want += cbf[s, codes[(s * rows + r) * nv + v], i]
                assert got[r, 8 * v + i] == want
    # the same weights as the position-major reader on the transposed planes
    pm = codes.reshape(3, rows, nv).transpose(0, 2, 1).copy()
    np.testing.assert_array_equal(got, oracle.rvq3_matrix(pm, cb, rows, K))
    # a whole expert: row-major record = position-major record with every plane transposed
    d, ff = 64, 96
    rec = si.rvq3_record(7, 1, d, ff)
    cbs = np.stack([si.normal(7, 16 + s, 0.02 / (s + 1), 256 * 8, "f16") for s in range(3)]).reshape(3, 256, 8)
    x = npref.to_f64(si.normal(7, 1, 1.0, d, "bf16"))
    parts, o = [], 0
    for rws, kk in ((ff, d), (ff, d), (d, ff)):
        n = 3 * rws * (kk // 8)
        parts.append(rec[o:o + n].reshape(3, rws, kk // 8).transpose(0, 2, 1).reshape(-1))
        o += n
    y_rm = oracle.expert_rvq3_rowmajor(x, rec, cbs, cbs, cbs, d, ff)
    y_pm = oracle.expert_rvq3(x, np.concatenate(parts), cbs, cbs, cbs, d, ff)
    np.testing.assert_array_equal(y_rm, y_pm)


def test_record_sizes_match_page_figures():
    with open(os.path.join(GOLDEN, "page_figures.json")) as f:
        pf = json.load(f)
    d, ff = pf["latent_shape"]["d"], pf["latent_shape"]["ff"]
    b = oracle.mxfp4_record_bytes(d, ff)
    assert b == 17_547_264
    assert round(b / 1e6, 2) == pf["mxfp4_expert_mb"]["value"]
    assert round(b / 1e6, 1) == pf["mxfp4_expert_mb_lazylora"]["value"]
    assert round(b * pf["mxfp4_layer_gb"]["experts"] / 1e9, 1) == pf["mxfp4_layer_gb"]["value"]
    assert pf["routed_experts_total"]["layers"] * pf["routed_experts_total"]["experts_per_layer"] == \
        pf["routed_experts_total"]["value"]
    rv = oracle.rvq3_record_bytes(d, ff)
    assert rv * 8 / (3 * d * ff) == pf["rvq3_bits_per_weight"]["value"]
    assert rv == 12_386_304
    # the generator's record layout agrees with the oracle's
    assert si.mxfp4_record_size(d, ff) == b and si.rvq3_record_size(d, ff) == rv


# ----------------------------------------------------------------------------- record checksum

def test_crc32_published_check_value_and_empty_input():
    # the catalogue check value of CRC-32/ISO-HDLC (the zlib/PNG CRC) over "123456789"
    assert oracle.crc32(b"123456789") == 0xCBF43926
    assert oracle.crc32(b"") == 0
    assert oracle.crc32(b"\x00") == 0xD202EF8D


def test_crc32_matches_zlib_on_random_buffers():
    import zlib
    rng = np.random.default_rng(7)
    for n in (1, 3, 16, 63, 64, 65, 1000, 4096, 52224):
        buf = rng.integers(0, 256, n, dtype=np.uint8)
        assert oracle.crc32(buf) == zlib.crc32(buf.tobytes()), n


def test_crc32_of_a_record_changes_with_any_single_bit():
    r = si.LayerRecipe("c", d=64, ff=64, E=2, k=1, T=1, x_dtype="f32", w_dtype="f32", seed=3)
    rec = si.layer_record(r, 1)
    c0 = oracle.crc32(rec)
    rng = np.random.default_rng(1)
    for pos in rng.integers(0, rec.size, 8):
        bad = rec.copy()
        bad[pos] ^= np.uint8(1 << int(rng.integers(0, 8)))
        assert oracle.crc32(bad) != c0


# ----------------------------------------------------------------------------- router

def _tiny_xw(T=12, d=64, E=24, seed=5, dt="bf16"):
    x = si.normal(seed, 1, 1.0, T * d, dt).reshape(T, d)
    W = si.normal(seed, 2, 1 / math.sqrt(d), E * d, dt).reshape(E, d)
    return x, W


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_router_logits_match_numpy_matmul(dt):
    # catches a transposed W or a dropped bias
    x, W = _tiny_xw(dt=dt)
    bias = si.normal(9, 3, 0.5, W.shape[0], "f32")
    logits, idx, g = oracle.router(x, W, bias, 5)
    ref = npref.to_f64(x) @ npref.to_f64(W).T + bias.astype(np.float64)[None]
    scale = np.abs(npref.to_f64(x)) @ np.abs(npref.to_f64(W)).T
    assert np.all(np.abs(logits - ref) <= 1e-13 * (scale + 1))


def test_router_one_hot_rows_select_coordinates():
    # W = identity rows: logit e is exactly x[e]
    T, d = 4, 32
    x = si.normal(2, 1, 1.0, T * d, "f32").reshape(T, d)
    W = np.eye(d, dtype=np.float32)
    logits, idx, g = oracle.router(x, W, None, 3)
    np.testing.assert_array_equal(logits, x.astype(np.float64))
    np.testing.assert_array_equal(idx, npref.topk_sorted(x.astype(np.float64), 3))


def test_topk_matches_full_sort_every_token():
    x, W = _tiny_xw(T=64, E=40)
    logits, idx, g = oracle.router(x, W, None, 7)
    np.testing.assert_array_equal(idx, npref.topk_sorted(logits, 7))


def test_topk_exact_ties_go_to_lower_index():
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.0],
                       [5.0, 5.0, 5.0, 5.0, 5.0, 5.0],
                       [0.0, -1.0, 0.0, 7.0, 7.0, -1.0]])
    idx, g = oracle.topk_gates(logits, 4)
    np.testing.assert_array_equal(idx, [[1, 2, 4, 3], [0, 1, 2, 3], [3, 4, 0, 2]])
    np.testing.assert_array_equal(idx, npref.topk_sorted(logits, 4))
    assert np.all(g[1] == 0.25)


def test_gates_sum_to_one_and_equal_renormalised_full_softmax():
    x, W = _tiny_xw(T=32, E=40)
    bias = si.zipf_bias(40)
    logits, idx, g = oracle.router(x, W, bias, 6)
    assert np.all(np.abs(g.sum(axis=1) - 1.0) <= 4e-16 * 6)
    ref = npref.gates_full_softmax(logits, idx)
    assert np.all(np.abs(g - ref) <= 1e-14 * ref)
    assert np.all(np.diff(g, axis=1) <= 0)  # ordered with the logits


def test_select_bias_mode_without_bias_or_with_uniform_bias_is_the_plain_router():
    x, W = _tiny_xw(T=16, E=30)
    l0, i0, g0 = oracle.router(x, W, None, 5)
    l1, i1, g1 = oracle.router(x, W, None, 5, bias_mode="select")
    np.testing.assert_array_equal(i1, i0)
    np.testing.assert_array_equal(g1, g0)
    # a bias equal for every expert moves no selection; the selection-only
    # gates ignore it, the additive ones cancel it in the softmax
    c = np.full(30, 2.5, dtype=np.float32)
    l2, i2, g2 = oracle.router(x, W, c, 5, bias_mode="select")
    np.testing.assert_array_equal(i2, i0)
    np.testing.assert_array_equal(g2, g0)
    np.testing.assert_array_equal(l2, l0 + 2.5)


def test_select_bias_forces_the_selection_and_gates_follow_the_unbiased_logits():
    # the bias lifts a fixed set of k experts 1000 (plus distinct offsets that
    # fix their order) above the rest: they are the selection whatever the
    # logits, and their gates are the softmax of the logits WITHOUT the bias,
    # i.e. g_a / g_b = exp(l_a - l_b) with l from a plain matmul
    T, d, E, k = 10, 64, 24, 4
    x, W = _tiny_xw(T=T, d=d, E=E)
    chosen = [17, 3, 22, 8]
    bias = np.zeros(E, dtype=np.float32)
    for r, e in enumerate(chosen):
        bias[e] = 1000.0 - 10.0 * r
    keys, idx, g = oracle.router(x, W, bias, k, bias_mode="select")
    assert np.all(idx == np.array(chosen)[None, :])
    plain = npref.to_f64(x) @ npref.to_f64(W).T
    for t in range(T):
        lsel = plain[t, chosen]
        for a in range(k):
            for b in range(k):
                assert g[t, a] / g[t, b] == pytest.approx(math.exp(lsel[a] - lsel[b]), rel=1e-12)
    assert np.all(np.abs(g.sum(axis=1) - 1.0) <= 1e-15 * k)
    # the offsets among the chosen experts change nothing in the selection-only
    # gates (they would, in the additive mode)
    bias2 = bias.copy()
    bias2[chosen] += np.array([0.0, 3.0, 1.0, 2.0], dtype=np.float32)
    _, idx2, g2 = oracle.router(x, W, bias2, k, bias_mode="select")
    _, _, g_add = oracle.router(x, W, bias2, k)
    np.testing.assert_array_equal(idx2, idx)
    np.testing.assert_array_equal(g2, g)
    assert np.max(np.abs(g_add - g)) > 0.1


def test_select_bias_gates_match_renormalised_full_softmax_of_plain_logits():
    x, W = _tiny_xw(T=32, E=40)
    bias = si.zipf_bias(40)
    keys, idx, g = oracle.router(x, W, bias, 6, bias_mode="select")
    plain = npref.to_f64(x) @ npref.to_f64(W).T
    np.testing.assert_array_equal(idx, npref.topk_sorted(plain + bias.astype(np.float64)[None], 6))
    ref = npref.gates_full_softmax(plain, idx)
    assert np.all(np.abs(g - ref) <= 1e-13 * ref)


# ----------------------------------------------------------------------------- bucketing

def test_bucket_matches_brute_force_scan():
    rng = np.random.default_rng(1)
    T, k, E = 37, 5, 23
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, pair_ids = oracle.bucket(idx, E)
    flat = idx.reshape(-1)
    exp_ids = []
    for e in range(E):  # O(E * T * k) scan, ascending pair id within each expert
        ids = [p for p in range(T * k) if flat[p] == e]
        assert counts[e] == len(ids)
        exp_ids += ids
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    np.testing.assert_array_equal(pair_ids, exp_ids)
    assert sorted(pair_ids.tolist()) == list(range(T * k))
    assert npref.fnv1a64(pair_ids) == npref.fnv1a64(np.array(exp_ids, dtype=np.int32))


def test_bucket_rejects_out_of_range_expert():
    idx = np.array([[0, 5]], dtype=np.int32)
    with pytest.raises(RuntimeError):
        oracle.bucket(idx, 4)


# ----------------------------------------------------------------------------- expert FFN

def _const_record(d, ff, gate_code, gate_scale, rng):
    """Gate and up matrices constant (one code, one scale byte); down random."""
    cbytes, sbytes = ff * d // 2, ff * d // 32
    rec = []
    for _ in range(2):
        rec.append(np.full(cbytes, gate_code | (gate_code << 4), dtype=np.uint8))
        rec.append(np.full(sbytes, gate_scale, dtype=np.uint8))
    rec.append(rng.integers(0, 256, size=d * ff // 2, dtype=np.uint8))
    rec.append(rng.integers(118, 126, size=d * ff // 32, dtype=np.uint8))
    return np.concatenate(rec)


def test_expert_closed_form_constant_gate_up():
    # Wg = Wu = c * ones: g = u = c * sum(x); h = silu(g) * u for every row;
    # y_i = rowsum(Wd)_i * h.  Catches a transposed down matrix or act mix-up.
    d, ff = 64, 96
    rng = np.random.default_rng(0)
    rec = _const_record(d, ff, 2, 124, rng)  # code 2 = 1.0, c = 2^-3
    x = npref.to_f64(si.normal(4, 1, 1.0, d, "bf16"))
    c = 2.0 ** -3
    s = c * x.sum()
    h = s / (1.0 + math.exp(-s)) * s
    wd = npref.mxfp4_record_mats(rec, d, ff)[2]
    y = oracle.expert_mxfp4(x, rec, d, ff)
    ref = wd.sum(axis=1) * h
    assert np.all(np.abs(y - ref) <= 1e-12 * (np.abs(wd).sum(axis=1) * abs(h) + 1e-300))


def test_expert_all_zero_codes_give_zero():
    d, ff = 64, 64
    rec = np.zeros(oracle.mxfp4_record_bytes(d, ff), dtype=np.uint8)
    rec[:] = 0
    x = npref.to_f64(si.normal(1, 1, 1.0, d, "bf16"))
    assert np.all(oracle.expert_mxfp4(x, rec, d, ff) == 0.0)


@pytest.mark.parametrize("act", ["swiglu", "situ"])
def test_expert_mxfp4_matches_numpy(act):
    d, ff = 96, 64
    rec = si.mxfp4_record(3, 2, d, ff, 119, 125)
    x = npref.to_f64(si.normal(3, 1, 1.0, d, "bf16"))
    y = oracle.expert_mxfp4(x, rec, d, ff, act)
    ref = npref.expert(x, npref.mxfp4_record_mats(rec, d, ff), act)
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_expert_rvq3_matches_numpy():
    d, ff = 64, 96
    rec = si.rvq3_record(3, 4, d, ff)
    cb = [si.normal(3, 16 + s, 0.02 / (s + 1), 256 * 8, "f16") for s in range(3)]
    cbs = np.stack(cb).reshape(3, 256, 8)
    x = npref.to_f64(si.normal(3, 1, 1.0, d, "bf16"))
    y = oracle.expert_rvq3(x, rec, cbs, cbs, cbs, d, ff)
    ref = npref.expert(x, npref.rvq3_record_mats(rec, [cbs, cbs, cbs], d, ff))
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_situ_limits():
    # small arguments: SiTU -> silu(g) * u (tanh(z) ~ z); saturated gate: -> 100 tanh(u/25)
    for g, u in [(1e-3, 2e-3), (-2e-3, 1e-3)]:
        sw = oracle.act(g, u, "swiglu")
        st = oracle.act(g, u, "situ")
        assert abs(st - sw) <= 1e-6 * abs(sw)
    for u in (-30.0, 1.0, 80.0):
        assert abs(oracle.act(200.0, u, "situ") - 100.0 * math.tanh(u / 25.0)) <= 1e-12 * 100
    assert oracle.act(-200.0, 3.0, "situ") == pytest.approx(0.0, abs=1e-80)
    # SwiGLU against scipy's logistic
    from scipy.special import expit
    for g, u in [(0.3, -1.2), (-4.0, 2.0), (9.0, 0.5)]:
        assert oracle.act(g, u) == pytest.approx(g * expit(g) * u, rel=1e-15)


# ----------------------------------------------------------------------------- combine / whole layer

def _tiny_layer(seed=0, T=6, d=64, ff=64, E=12, k=3, quant="mxfp4"):
    r = si.LayerRecipe("t", d=d, ff=ff, E=E, k=k, T=T, x_dtype="f32", w_dtype="f32", seed=seed, scale_lo=119,
                       scale_hi=125, quant=quant)
    x = si.layer_x(r)
    W = si.layer_router_w(r)
    recs = [si.layer_record(r, e) for e in range(E)]
    return r, x, W, recs


def test_layer_matches_numpy_chain():
    r, x, W, recs = _tiny_layer()
    idx, g, y, out = oracle.layer_forward(x, W, None, r.d, r.ff, r.E, r.k, recs)
    logits, idx_ref, g_ref, delta_ref = npref.layer(x, W, None, r.k,
                                                    lambda e: npref.mxfp4_record_mats(recs[e], r.d, r.ff))
    np.testing.assert_array_equal(idx, idx_ref)
    assert np.all(np.abs(g - g_ref) <= 1e-14 * g_ref)
    assert np.max(np.abs(y - delta_ref)) <= 1e-12 * np.max(np.abs(delta_ref))
    np.testing.assert_allclose(out, x.astype(np.float64) + y, rtol=0, atol=1e-12 * np.max(np.abs(out)))


def test_layer_rvq3_matches_numpy_chain():
    r, x, W, recs = _tiny_layer(quant="rvq3", seed=4)
    cbs = si.layer_codebooks(r)
    idx, g, y, out = oracle.layer_forward(x, W, None, r.d, r.ff, r.E, r.k, recs, quant="rvq3",
                                          codebooks=(cbs, cbs, cbs))
    _, idx_ref, g_ref, delta_ref = npref.layer(x, W, None, r.k,
                                               lambda e: npref.rvq3_record_mats(recs[e], [cbs] * 3, r.d, r.ff))
    np.testing.assert_array_equal(idx, idx_ref)
    assert np.max(np.abs(y - delta_ref)) <= 1e-12 * np.max(np.abs(delta_ref))


def test_layer_select_bias_and_shared_experts_match_numpy_chain():
    E, S = 12, 2
    r, x, W, recs = _tiny_layer(E=E + S, seed=6)
    bias = si.zipf_bias(E)
    W = W[:E]
    mats = lambda e: npref.mxfp4_record_mats(recs[e], r.d, r.ff)
    for mode in ("logit", "select"):
        idx, g, y, out = oracle.layer_forward(x, W, bias, r.d, r.ff, E, r.k, recs, n_shared=S, bias_mode=mode)
        _, idx_ref, g_ref, delta_ref = npref.layer(x, W, bias, r.k, mats, bias_mode=mode, n_shared=S)
        np.testing.assert_array_equal(idx, idx_ref)
        assert np.all(np.abs(g - g_ref) <= 1e-13 * g_ref)
        assert np.max(np.abs(y - delta_ref)) <= 1e-12 * np.max(np.abs(delta_ref))


def test_shared_experts_add_their_unweighted_outputs():
    E, S = 12, 2
    r, x, W, recs = _tiny_layer(E=E + S, seed=8)
    W = W[:E]
    idx0, g0, y0, _ = oracle.layer_forward(x, W, None, r.d, r.ff, E, r.k, recs[:E])
    idx, g, y, out = oracle.layer_forward(x, W, None, r.d, r.ff, E, r.k, recs, n_shared=S)
    np.testing.assert_array_equal(idx, idx0)
    np.testing.assert_array_equal(g, g0)
    for t in range(r.T):
        xt = x[t].astype(np.float64)
        shared = sum(oracle.expert_mxfp4(xt, recs[E + s], r.d, r.ff) for s in range(S))
        np.testing.assert_allclose(y[t] - y0[t], shared, rtol=0, atol=1e-12 * np.max(np.abs(y[t])))
    # a shared expert whose codes are all zero adds exactly nothing
    zero = recs[E].copy()
    zero[:] = 0
    _, _, y1, _ = oracle.layer_forward(x, W, None, r.d, r.ff, E, r.k, recs[:E] + [zero], n_shared=1)
    np.testing.assert_array_equal(y1, y0)
    # a missing shared record is an error, as for a routed one
    with pytest.raises(RuntimeError):
        oracle.layer_forward(x, W, None, r.d, r.ff, E, r.k, recs[:E] + [None], n_shared=1)


def test_one_hot_gate_reproduces_single_expert():
    # a bias that puts one expert 2000 above the rest: its gate is exactly 1 and
    # every other selected gate underflows to exactly 0 in fp64
    r, x, W, recs = _tiny_layer()
    bias = np.zeros(r.E, dtype=np.float32)
    bias[7] = 2000.0
    idx, g, y, out = oracle.layer_forward(x, W, bias, r.d, r.ff, r.E, r.k, recs)
    assert np.all(idx[:, 0] == 7) and np.all(g[:, 0] == 1.0) and np.all(g[:, 1:] == 0.0)
    for t in range(r.T):
        np.testing.assert_array_equal(y[t], oracle.expert_mxfp4(x[t].astype(np.float64), recs[7], r.d, r.ff))


def test_zero_weight_experts_contribute_nothing_even_if_nan():
    r, x, W, recs = _tiny_layer()
    bias = np.zeros(r.E, dtype=np.float32)
    bias[7] = 2000.0
    idx, g, y, out = oracle.layer_forward(x, W, bias, r.d, r.ff, r.E, r.k, recs)
    poisoned = list(recs)
    for e in set(idx[:, 1:].reshape(-1).tolist()) - {7}:
        rec = recs[e].copy()
        cbytes, sbytes = r.ff * r.d // 2, r.ff * r.d // 32
        rec[cbytes:cbytes + sbytes] = 255  # NaN scales
        poisoned[e] = rec
    idx2, g2, y2, out2 = oracle.layer_forward(x, W, bias, r.d, r.ff, r.E, r.k, poisoned)
    assert np.all(np.isfinite(y2))
    np.testing.assert_array_equal(y2, y)


def test_combine_without_residual_is_the_weighted_sum():
    rng = np.random.default_rng(2)
    T, k, d = 3, 4, 8
    yp = rng.standard_normal((T * k, d))
    g = rng.random((T, k))
    g[1, 2] = 0.0
    yp[1 * k + 2] = np.nan  # skipped because its gate is 0
    out = oracle.combine(None, yp, g, k)
    for t in range(T):
        ref = sum(g[t, j] * yp[t * k + j] for j in range(k) if g[t, j] != 0)
        np.testing.assert_allclose(out[t], ref, rtol=1e-15, atol=1e-15)
    xr = rng.standard_normal((T, d))
    np.testing.assert_allclose(oracle.combine(xr, yp, g, k) - xr, out, rtol=1e-14, atol=1e-14)


def test_missing_routed_expert_is_an_error():
    r, x, W, recs = _tiny_layer()
    idx, g, y, out = oracle.layer_forward(x, W, None, r.d, r.ff, r.E, r.k, recs)
    missing = list(recs)
    missing[int(idx[0, 0])] = None
    with pytest.raises(RuntimeError):
        oracle.layer_forward(x, W, None, r.d, r.ff, r.E, r.k, missing)


def test_token_mask_and_threads_do_not_change_results():
    r, x, W, recs = _tiny_layer(T=8)
    idx, g, y, out = oracle.layer_forward(x, W, None, r.d, r.ff, r.E, r.k, recs)
    mask = np.array([1, 0, 1, 0, 0, 1, 0, 0], dtype=np.uint8)
    idx2, g2, y2, out2 = oracle.layer_forward(x, W, None, r.d, r.ff, r.E, r.k, recs, token_mask=mask, nthreads=4)
    np.testing.assert_array_equal(idx2, idx)
    np.testing.assert_array_equal(y2[mask == 1], y[mask == 1])
    assert np.all(np.isnan(y2[mask == 0]))


def test_partial_deltas_over_expert_ranges_sum_to_full():
    r, x, W, recs = _tiny_layer(T=8, E=12)
    idx, g, y, out = oracle.layer_forward(x, W, None, r.d, r.ff, r.E, r.k, recs)
    a = oracle.partial_delta(x, idx, g, r.d, r.ff, r.k, recs, 0, 5)
    b = oracle.partial_delta(x, idx, g, r.d, r.ff, r.k, recs, 5, 12)
    np.testing.assert_allclose(a + b, y, rtol=0, atol=1e-12 * np.max(np.abs(y)))


# ---- latent projections (LazyLoRA README, "The engine": the experts work in a
# 3584-wide latent space between projections from and back to the model width)

def _bf16_of(a32):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("xdt,wdt", [("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32")])
def test_project_matches_numpy(xdt, wdt):
    T, K, N = 3, 160, 96
    x = si.normal(21, 1, 1.0, T * K, xdt).reshape(T, K)
    W = si.normal(21, 2, 0.05, N * K, wdt).reshape(N, K)
    y = oracle.project(x, W)
    xf = npref.to_f64(x) if xdt == "bf16" else x.astype(np.float64)
    wf = npref.to_f64(W) if wdt == "bf16" else W.astype(np.float64)
    ref = xf @ wf.T
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(xf)) * np.max(np.abs(wf)) * K
    # row n of W against token t, element by element: a transposed W would differ
    assert y.shape == (T, N) and abs(y[1, 7] - sum(wf[7] * xf[1])) <= 1e-12


def test_round_bf16_is_round_to_nearest_even():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.normal(0, 1, 2000), rng.normal(0, 1e-38, 200), rng.normal(0, 1e38, 200)]).astype(np.float32)
    # exact ties: a bf16 value plus half its spacing, with even and odd last bits
    base = np.array([1.0, 1.0078125, 3.0, 255.0, -1.0078125], dtype=np.float32)
    ties = (base.astype(np.float64) + np.abs(base).astype(np.float64) * 2.0 ** -8).astype(np.float32)
    v = np.concatenate([v, ties, np.array([0.0, -0.0, 3.4e38, -3.4e38, 1e-45], dtype=np.float32)])
    got = oracle.round_bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, _bf16_of(v))
    assert oracle.round_bf16(np.array([np.nan]))[0] & 0x7FFF > 0x7F80
    assert list(oracle.round_bf16(np.array([1.00390625, 1.01171875]))) == [0x3F80, 0x3F82]  # ties to even


def _latent_case(D, seed, perm=None, identity=False):
    r = si.LayerRecipe("latent_tiny", d=64, ff=64, E=8, k=2, T=3, seed=seed, x_dtype="bf16", w_dtype="bf16",
                       scale_lo=119, scale_hi=125)
    recs = [si.layer_record(r, e) for e in range(r.E)]
    W = si.layer_router_w(r)
    x = si.normal(seed, 90, 1.0, r.T * D, "bf16").reshape(r.T, D)
    if identity:
        w_in = np.zeros((r.d, D), dtype=np.uint16)
        w_in[np.arange(r.d), np.arange(r.d) if perm is None else perm] = 0x3F80  # 1.0
        w_out = np.ascontiguousarray(w_in.T)
    else:
        w_in = si.normal(seed, 91, 1.0 / np.sqrt(D), r.d * D, "bf16").reshape(r.d, D)
        w_out = si.normal(seed, 92, 1.0 / np.sqrt(r.d), D * r.d, "bf16").reshape(D, r.d)
    return r, recs, W, x, w_in, w_out


def test_latent_identity_projection_is_the_plain_layer():
    r, recs, W, x, w_in, w_out = _latent_case(64, 31, identity=True)
    z, out = oracle.latent_forward(x, w_in, w_out, W, None, r.d, r.ff, r.E, r.k, recs)
    np.testing.assert_array_equal(z, x)
    _, _, _, o = oracle.layer_forward(x, W, None, r.d, r.ff, r.E, r.k, recs)
    np.testing.assert_array_equal(out, o)


def test_latent_one_hot_projection_selects_inputs():
    D = 96
    perm = np.random.default_rng(3).permutation(D)[:64]
    r, recs, W, x, w_in, w_out = _latent_case(D, 32, perm=perm, identity=True)
    z, out = oracle.latent_forward(x, w_in, w_out, W, None, r.d, r.ff, r.E, r.k, recs)
    np.testing.assert_array_equal(z, x[:, perm])  # z[t][n] = x[t][perm[n]]
    _, _, y, _ = oracle.layer_forward(z, W, None, r.d, r.ff, r.E, r.k, recs)
    want = npref.to_f64(x).copy()
    want[:, perm] += y  # W_out scatters the latent delta back to the selected inputs
    np.testing.assert_array_equal(out, want)


def test_latent_layer_matches_numpy_chain():
    D = 80
    r, recs, W, x, w_in, w_out = _latent_case(D, 33)
    z, out = oracle.latent_forward(x, w_in, w_out, W, None, r.d, r.ff, r.E, r.k, recs)
    zr = npref.to_f64(x) @ npref.to_f64(w_in).T
    np.testing.assert_array_equal(z, _bf16_of(zr.astype(np.float32)))  # no value sits at a rounding tie here
    _, _, y, _ = oracle.layer_forward(z, W, None, r.d, r.ff, r.E, r.k, recs)
    ref = npref.to_f64(x) + y @ npref.to_f64(w_out).T
    assert np.max(np.abs(out - ref)) <= 1e-12 * np.max(np.abs(ref))
