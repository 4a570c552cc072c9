"""GPU record check: the CRC-32 of expert records computed by the library
against the oracle's bit-at-a-time CRC (pinned to zlib and the published check
value), and the check's reports of a changed, missing or misaligned record."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from quantized_expert_ffn_score_gb300 import build, moe
    build.build()
    return moe


@pytest.fixture(scope="module")
def ctx(moe):
    c = moe.Context(0)
    yield c
    c.close()


def _crc(moe, ctx, ptrs, record_bytes, expected=None):
    n = len(ptrs)
    recs = torch.tensor(ptrs, dtype=torch.int64, device="cuda")
    out = torch.zeros(n, dtype=torch.int32, device="cuda")
    ws = moe.workspace(moe.records_check_ws_bytes(n, record_bytes))
    exp = None if expected is None else torch.from_numpy(np.asarray(expected, dtype=np.uint32).view(np.int32)).cuda()
    moe.moe_records_check(ctx, recs, n, record_bytes, ws, expected=exp, crc_out=out)
    return out.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("record_bytes", [16, 48, 1632, 4096, 131072, 131088, 52224, 3 * 131072 + 1632])
def test_crc_of_random_records_matches_oracle(moe, ctx, record_bytes):
    # sizes below one segment, at and just past a segment boundary, several
    # segments with a ragged head; three records at a 16-byte (not 256-byte) stride
    rng = np.random.default_rng(record_bytes)
    n = 3
    host = rng.integers(0, 256, n * record_bytes + 16, dtype=np.uint8)
    dev = torch.from_numpy(host).cuda()
    base = dev.data_ptr() + 16 - dev.data_ptr() % 16 if dev.data_ptr() % 16 else dev.data_ptr()
    off = base - dev.data_ptr()
    ptrs = [base + e * record_bytes for e in range(n)]
    got = _crc(moe, ctx, ptrs, record_bytes)
    ctx.check()
    for e in range(n):
        ref = oracle.crc32(host[off + e * record_bytes:off + (e + 1) * record_bytes])
        assert int(got[e]) == ref, (record_bytes, e)


def test_crc_of_the_tiny_bank_and_a_sample_of_the_k3_bank(moe, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    for name, sample in (("tiny", range(16)), ("k3_mxfp4_decode", (0, 417, 895))):
        r = si.get_workload(name)
        layer = synthetic.device_layer(r)
        nbytes = si.record_size(r)
        ptrs = [layer.bank.data_ptr() + e * layer.stride for e in range(r.E)]
        got = _crc(moe, ctx, ptrs, nbytes)
        ctx.check()
        for e in sample:
            assert int(got[e]) == oracle.crc32(si.layer_record(r, e)), (name, e)
        del layer


def test_check_reports_a_changed_missing_or_misaligned_record(moe, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = si.get_workload("tiny")
    layer = synthetic.device_layer(r)
    nbytes = si.record_size(r)
    ptrs = [layer.bank.data_ptr() + e * layer.stride for e in range(r.E)]
    good = _crc(moe, ctx, ptrs, nbytes)
    ctx.check()
    _crc(moe, ctx, ptrs, nbytes, expected=good)  # all records as expected
    ctx.check()
    layer.bank[5 * layer.stride + 1000] ^= 1  # one bit of record 5
    got = _crc(moe, ctx, ptrs, nbytes, expected=good)
    with pytest.raises(moe.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_BAD_RECORD" and ei.value.detail == 5
    assert got[5] != good[5] and np.array_equal(np.delete(got, 5), np.delete(good, 5))
    layer.bank[5 * layer.stride + 1000] ^= 1
    missing = list(ptrs)
    missing[9] = 0
    _crc(moe, ctx, missing, nbytes, expected=good)
    with pytest.raises(moe.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_MISSING_EXPERT" and ei.value.detail == 9
    shifted = list(ptrs)
    shifted[3] += 8  # not 16-byte aligned: reported, never read
    got = _crc(moe, ctx, shifted, nbytes)
    with pytest.raises(moe.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_BAD_RECORD" and ei.value.detail == 3 and got[3] == 0
    ctx.check()
    with pytest.raises(moe.MoeError) as ei:  # size not a multiple of 16
        _crc(moe, ctx, ptrs, nbytes - 8)
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
