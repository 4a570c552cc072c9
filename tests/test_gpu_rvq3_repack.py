"""moe_rvq3_repack: RVQ3 records whose code planes are stored row by row
([3][rows][K/8] per matrix) converted to the position-major layout the RVQ3
kernels read, through the C ABI.

The converted bytes must equal the transposed planes exactly (index work, so
bit-exact), and a layer whose bank was given row-major and converted must
match the oracle reading the row-major records directly: routing bit-exact,
outputs within 2e-3 x RMS.  A NULL record and an in-place conversion are
reported on the error word by record index."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

MID = si.LayerRecipe("rvq3_rowmajor_mid", d=1024, ff=576, E=24, k=4, T=11, seed=61, quant="rvq3")
# ff / 8 = 16 positions: the down planes' tiles are ragged in the position axis
SMALL = si.LayerRecipe("rvq3_rowmajor_small", d=256, ff=128, E=6, k=2, T=5, seed=62, quant="rvq3")


@pytest.fixture(scope="module")
def lib():
    from quantized_expert_ffn_score_gb300 import build, moe
    build.build()
    return moe


@pytest.fixture()
def ctx(lib):
    c = lib.Context(0)
    yield c
    c.close()


def _converted_layer(moe, ctx, r):
    """The recipe's record bytes taken as row-major records, converted into a
    second bank; returns (layer on the converted bank, row-major bank)."""
    from quantized_expert_ffn_score_gb300 import synthetic
    layer = synthetic.device_layer(r)  # bank bytes: the seeded records
    n = r.E + r.n_shared
    src_bank = layer.bank
    dst_bank = torch.full_like(src_bank, 0xAB)
    src = torch.tensor([src_bank.data_ptr() + e * layer.stride for e in range(n)], dtype=torch.int64, device="cuda")
    dst = torch.tensor([dst_bank.data_ptr() + e * layer.stride for e in range(n)], dtype=torch.int64, device="cuda")
    moe.moe_rvq3_repack(ctx, src, dst, n, r.d, r.ff)
    ctx.check()
    conv = moe.Layer(r.d, r.ff, r.E, r.k, layer.router_w, dst, quant="rvq3", act=r.act,
                     router_bias=layer.router_bias, codebooks=layer.codebooks, keep=[dst_bank, layer],
                     n_shared=r.n_shared, bias_mode=r.bias_mode)
    conv.recipe = r
    conv.bank, conv.stride = dst_bank, layer.stride
    return conv, layer


@pytest.mark.parametrize("r", [MID, SMALL], ids=["mid", "small"])
def test_converted_bytes_are_the_transposed_planes(lib, ctx, r):
    conv, layer = _converted_layer(lib, ctx, r)
    nbytes = si.record_size(r)
    for e in (0, r.E - 1):
        got = conv.bank[e * conv.stride:e * conv.stride + nbytes].cpu().numpy()
        rm = si.layer_record(r, e)
        want, o = [], 0
        for rows, K in ((r.ff, r.d), (r.ff, r.d), (r.d, r.ff)):
            n = 3 * rows * (K // 8)
            want.append(rm[o:o + n].reshape(3, rows, K // 8).transpose(0, 2, 1).reshape(-1))
            o += n
        np.testing.assert_array_equal(got, np.concatenate(want))


def _oracle_rowmajor_layer(r, xh):
    """Oracle routing, then every pair through the row-major expert reader, then the combine."""
    W = si.layer_router_w(r)
    logits, idx, g = oracle.router(xh, W, si.layer_bias(r), r.k, bias_mode=r.bias_mode)
    cb = si.layer_codebooks(r)
    x64 = gu.x_host_f64(xh)
    y = np.zeros((r.T * r.k, r.d))
    recs = si.layer_records(r, np.unique(idx))
    for p in range(r.T * r.k):
        y[p] = oracle.expert_rvq3_rowmajor(x64[p // r.k], recs[idx.reshape(-1)[p]], cb, cb, cb, r.d, r.ff,
                                           act_kind=r.act)
    delta = oracle.combine(None, y, g.reshape(-1), r.k)
    return logits, idx, g, delta


@pytest.mark.parametrize("r", [MID, SMALL], ids=["mid", "small"])
def test_layer_on_converted_bank_matches_oracle_on_row_major_records(lib, ctx, r):
    from quantized_expert_ffn_score_gb300 import synthetic
    conv, _ = _converted_layer(lib, ctx, r)
    x = synthetic.device_x(r)
    out, topk, gates, _ = gu.run_layer(lib, ctx, conv, x)
    xh = si.layer_x(r)
    logits, idx, g, delta = _oracle_rowmajor_layer(r, xh)
    gu.check_routing(topk, gates, idx, g, gu.gate_tolerance(r, xh, logits))
    d_gpu = out.astype(np.float64) - gu.x_host_f64(xh)
    err, rms = gu.rms_err(d_gpu, delta)
    gu.record_margin(r.name, err, rms, r.T)
    gu.assert_rms_close(d_gpu, delta, what=r.name)


@pytest.mark.slow
def test_k3_rvq3_decode_on_converted_bank(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = si.get_workload("k3_rvq3_decode_b1").with_(name="k3_rvq3_rowmajor_decode_b1")
    conv, layer = _converted_layer(lib, ctx, r)
    del layer
    x = synthetic.device_x(r)
    out, topk, gates, _ = gu.run_layer(lib, ctx, conv, x)
    xh = si.layer_x(r)
    logits, idx, g, delta = _oracle_rowmajor_layer(r, xh)
    gu.check_routing(topk, gates, idx, g, gu.gate_tolerance(r, xh, logits))
    d_gpu = out.astype(np.float64) - gu.x_host_f64(xh)
    err, rms = gu.rms_err(d_gpu, delta)
    gu.record_margin(r.name, err, rms, r.T)
    gu.assert_rms_close(d_gpu, delta, what=r.name)


def test_null_and_in_place_records_are_reported(lib, ctx):
    r = SMALL
    nbytes = si.record_size(r)
    bank = torch.zeros(4 * nbytes, dtype=torch.uint8, device="cuda")
    out = torch.zeros(4 * nbytes, dtype=torch.uint8, device="cuda")
    base, obase = bank.data_ptr(), out.data_ptr()
    src = torch.tensor([base, 0, base + 2 * nbytes, base + 3 * nbytes], dtype=torch.int64, device="cuda")
    dst = torch.tensor([obase, obase + nbytes, obase + 2 * nbytes, obase + 3 * nbytes], dtype=torch.int64,
                       device="cuda")
    lib.moe_rvq3_repack(ctx, src, dst, 4, r.d, r.ff)
    with pytest.raises(lib.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_MISSING_EXPERT" and ei.value.detail == 1
    dst_inplace = src.clone()
    dst_inplace[1] = obase + nbytes
    lib.moe_rvq3_repack(ctx, src[2:], dst_inplace[2:], 2, r.d, r.ff)  # both records converted in place
    with pytest.raises(lib.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_INVALID_ARG" and ei.value.detail in (0, 1)
    with pytest.raises(lib.MoeError) as ei:
        lib.moe_rvq3_repack(ctx, src, dst, 4, 100, r.ff)  # d not a multiple of 32
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    lib.moe_rvq3_repack(ctx, src, dst, 0, r.d, r.ff)  # n = 0: nothing to do
    ctx.check()
