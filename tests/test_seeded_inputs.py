"""The seeded input generator (host side; the device side is checked in test_gpu_inputs.py)."""
import numpy as np
import torch

import seeded_inputs as si


def test_normal_moments_and_offsets():
    x = si.normal(0, 1, 1.0, 400_000, "f32")
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.abs(x).max() <= 6.0
    a = si.normal(5, 7, 0.3, 1000, "f32")
    b = si.normal(5, 7, 0.3, 300, "f32", offset=700)
    np.testing.assert_array_equal(a[700:], b)
    assert not np.array_equal(si.normal(5, 8, 0.3, 1000, "f32"), a)  # streams differ
    assert not np.array_equal(si.normal(6, 7, 0.3, 1000, "f32"), a)  # seeds differ


def test_f16_and_bf16_rounding_match_library_rne():
    for sigma in (1e-6, 3e-5, 0.02, 1.0, 3e4, 1e5):
        f = si.normal(3, 5, sigma, 50_000, "f32")
        h = si.normal(3, 5, sigma, 50_000, "f16")
        with np.errstate(over="ignore"):
            np.testing.assert_array_equal(f.astype(np.float16).view(np.uint16), h)
        b = si.normal(3, 5, sigma, 50_000, "bf16")
        tb = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(tb, b)


def test_mxfp4_record_regions():
    d, ff = 256, 128
    rec = si.mxfp4_record(0, 3, d, ff, 119, 125)
    assert rec.size == si.mxfp4_record_size(d, ff) == 52_224
    cb, sb = ff * d // 2, ff * d // 32
    o = 0
    for rows, K in ((ff, d), (ff, d), (d, ff)):
        codes = rec[o:o + rows * K // 2]
        o += rows * K // 2
        scales = rec[o:o + rows * K // 32]
        o += rows * K // 32
        assert scales.min() >= 119 and scales.max() <= 125
        assert len(np.unique(scales)) == 7
        nib = np.concatenate([codes & 15, codes >> 4])
        counts = np.bincount(nib, minlength=16)
        assert counts.min() > 0.8 * nib.size / 16
    part = si.mxfp4_record(0, 3, d, ff, 119, 125, offset=cb - 8, n=40)
    np.testing.assert_array_equal(part, rec[cb - 8:cb + 32])
    assert not np.array_equal(si.mxfp4_record(0, 4, d, ff, 119, 125), rec)


def test_rvq3_record_and_codebooks():
    r = si.get_workload("k3_rvq3_decode_b1")
    assert si.rvq3_record_size(r.d, r.ff) == 12_386_304
    part = si.rvq3_record(r.seed, 5, r.d, r.ff, offset=1000, n=5000)
    assert part.dtype == np.uint8 and len(np.unique(part)) > 250
    cb = si.layer_codebooks(r)
    vals = cb.view(np.float16).astype(np.float64)
    for s in range(3):
        assert abs(vals[s].std() - 0.02 / (s + 1)) < 0.1 * 0.02 / (s + 1)


def test_zipf_bias():
    b = si.zipf_bias(896)
    assert b[0] == 0.0 and b.dtype == np.float32
    assert np.all(np.diff(b) < 0)
    assert abs(b[895] - (-np.log(896))) < 1e-6
