"""The streaming GEMV pair of the MXFP4 expert FFN (selected with
moe_ctx_set_mxfp4_kernel(MOE_MXFP4_GEMV)) on calls of many tokens, against the
fp64 oracle through the C ABI.  By default only one-token calls run it; here
it also takes buckets of up to a few hundred tokens, which it serves in passes
of 8 tokens (the warp-level MMA's N) over each staged weight tile.

Cases: a Zipf-skewed router (one bucket of many 8-token passes with a ragged
last pass, small buckets of one pass), every bucket about 50 tokens with the
last expert's bucket reaching the end of the slot range, SiTU, the standalone
expert call against the oracle's per-pair outputs, and a missing expert
reported on the error word."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

# Zipf(1) bias over 24 experts: buckets from 1 token to a few hundred
ZIPF = si.LayerRecipe("gemv_zipf", d=512, ff=512, E=24, k=4, T=300, seed=41, bias="zipf", scale_lo=118, scale_hi=121)
# 8 experts, 2 of them per token: every bucket ~50 tokens, the last one non-empty
UNIFORM = si.LayerRecipe("gemv_uniform", d=256, ff=256, E=8, k=2, T=203, seed=42)


@pytest.fixture(scope="module")
def lib():
    from quantized_expert_ffn_score_gb300 import build, moe
    build.build()
    return moe


@pytest.fixture()
def ctx(lib):
    c = lib.Context(0)
    c.mxfp4_kernel = "gemv"
    yield c
    c.close()


def test_zipf_buckets_in_many_passes(lib, ctx):
    _, counts = gu.full_check(lib, ctx, ZIPF)
    assert counts.max() > 16 * 8, "needs a bucket of many 8-token passes"
    assert np.any((counts > 8) & (counts % 8 != 0)), "needs a ragged last pass"
    assert np.any((counts > 0) & (counts <= 8)), "needs one-pass buckets too"


def test_uniform_buckets_last_expert_at_end_of_slots(lib, ctx):
    _, counts = gu.full_check(lib, ctx, UNIFORM)
    assert counts[-1] > 0 and counts.min() > 8


def test_situ(lib, ctx):
    gu.full_check(lib, ctx, ZIPF.with_(act="situ", seed=43, T=120))


def test_standalone_expert_call_matches_oracle_pairs(lib, ctx):
    import oracle
    from quantized_expert_ffn_score_gb300 import synthetic
    r = ZIPF
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    topk = torch.empty((r.T, r.k), dtype=torch.int32, device="cuda")
    gates = torch.empty((r.T, r.k), dtype=torch.float32, device="cuda")
    lib.moe_route_topk(ctx, x, layer.router_w, layer.router_bias, r.k, topk, gates,
                       lib.workspace(lib.route_topk_ws_bytes(r.T, r.d, r.E, r.k)))
    counts = torch.empty(r.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(r.E + 1, dtype=torch.int32, device="cuda")
    pairs = torch.empty(r.T * r.k, dtype=torch.int32, device="cuda")
    lib.moe_bucket_tokens(ctx, topk, r.E, counts, offsets, pairs, lib.workspace(lib.bucket_tokens_ws_bytes(r.T, r.k,
                                                                                                          r.E)))
    y = torch.full((r.T * r.k, r.d), float("nan"), dtype=torch.float32, device="cuda")
    lib.moe_expert_ffn_mxfp4(ctx, x, r.k, layer, offsets, pairs, y,
                             lib.workspace(lib.expert_ffn_ws_bytes(r.T, r.k, r.d, r.ff, r.E)))
    ctx.check()
    y = y.cpu().numpy().astype(np.float64)
    # the oracle's per-pair outputs (ungated): y_pairs[p] = expert(topk[p]) applied to x[p // k]
    xh = si.layer_x(r)
    _, idx, _ = oracle.router(xh, si.layer_router_w(r), si.layer_bias(r), r.k)
    ref = np.empty_like(y)
    for e in np.unique(idx):
        rec = si.layer_record(r, int(e))
        for p in np.nonzero(idx.reshape(-1) == e)[0]:
            ref[p] = oracle.expert_mxfp4(gu.x_host_f64(xh)[p // r.k], rec, r.d, r.ff, act_kind=r.act)
    gu.assert_rms_close(y, ref, what="GEMV expert call")


@pytest.mark.parametrize("static", [False, True])
def test_standalone_one_token_expert_call_matches_oracle(lib, ctx, static):
    # one token through the expert call itself: the per-token max |x| comes from
    # the launch just ahead of the expert kernels (not from a router two launches
    # earlier), so the one-token kernel must not stage x before its wait
    import oracle
    from quantized_expert_ffn_score_gb300 import synthetic
    r = ZIPF.with_(T=1, seed=41)
    layer = synthetic.device_layer(r)
    for call, offset in enumerate((0, 7)):  # two calls: the second must not see the first token's scale
        x = synthetic.device_x(r, token_offset=offset)
        topk = torch.empty((1, r.k), dtype=torch.int32, device="cuda")
        gates = torch.empty((1, r.k), dtype=torch.float32, device="cuda")
        lib.moe_route_topk(ctx, x, layer.router_w, layer.router_bias, r.k, topk, gates,
                           lib.workspace(lib.route_topk_ws_bytes(1, r.d, r.E, r.k)))
        counts = torch.empty(r.E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(r.E + 1, dtype=torch.int32, device="cuda")
        pairs = torch.empty(r.k, dtype=torch.int32, device="cuda")
        lib.moe_bucket_tokens(ctx, topk, r.E, counts, offsets, pairs,
                              lib.workspace(lib.bucket_tokens_ws_bytes(1, r.k, r.E)))
        y = torch.full((r.k, r.d), float("nan"), dtype=torch.float32, device="cuda")
        if static:
            lib.moe_expert_ffn_mxfp4_static(ctx, x, r.k, layer, offsets, pairs, y)
        else:
            lib.moe_expert_ffn_mxfp4(ctx, x, r.k, layer, offsets, pairs, y,
                                     lib.workspace(lib.expert_ffn_ws_bytes(1, r.k, r.d, r.ff, r.E)))
        ctx.check()
        xh = gu.x_host_f64(si.layer_x(r, T=1, token_offset=offset))
        idx = topk.cpu().numpy().reshape(-1)
        ref = np.stack([oracle.expert_mxfp4(xh[0], si.layer_record(r, int(e)), r.d, r.ff, act_kind=r.act) for e in idx])
        gu.assert_rms_close(y.cpu().numpy().astype(np.float64), ref, what=f"one-token expert call {call + 1}")


def test_missing_expert_is_reported(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = ZIPF
    layer = synthetic.device_layer(r, missing=[0])  # expert 0 has the largest bucket under the Zipf bias
    x = synthetic.device_x(r)
    out = torch.empty((r.T, r.d), dtype=torch.float32, device="cuda")
    lib.moe_layer_forward(ctx, layer, x, out, lib.workspace(lib.layer_forward_ws_bytes(layer, r.T)))
    with pytest.raises(lib.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_MISSING_EXPERT"
