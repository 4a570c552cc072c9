"""The block-scaled tensor-core kernel of the MXFP4 expert FFN (chosen by
default for bf16 activations with d, ff multiples of 512 and more than one
token; selected explicitly here) against the fp64 oracle, through the C ABI.

Cases: the smallest shapes (one scale group along K, a single padded n-tile,
ragged buckets), K split across CTAs with the last-arriver epilogue (few
pairs: every tile's K in parts of 512), several n-tiles (48 tokens for
gate/up, 40 for down) with ragged tails under a Zipf-skewed router, SiTU, the
standalone expert call against the oracle's per-pair outputs, agreement with
the GEMV kernel pair, one-token decode at the K3 shape, and a missing expert
reported on the error word.  The K3 prefill layers run on this kernel by default in
test_gpu_parity.py."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

# one scale group along K (d = ff = 512), 5 tokens: every n-tile padded from <= 8 tokens
SMALL = si.LayerRecipe("bs_small", d=512, ff=512, E=8, k=2, T=5, seed=51, scale_lo=118, scale_hi=121)
# 8 pairs over at most 8 experts: at most 64 tiles (half the CTAs or fewer), so every tile's K is
# split in two halves for two CTAs and finished by the one that arrives last
SPLIT = si.LayerRecipe("bs_split", d=1024, ff=1024, E=16, k=2, T=4, seed=52, scale_lo=118, scale_hi=121)
# one token routed to 3 experts: fewer pairs (3) than rows of an activation box (8)
FEWP = si.LayerRecipe("bs_fewp", d=512, ff=1024, E=8, k=3, T=1, seed=57, scale_lo=118, scale_hi=121)
# 37 tokens x 6 of 40 experts: n-tiles with ragged tails, d != ff
MID = si.LayerRecipe("bs_mid", d=1024, ff=512, E=40, k=6, T=37, seed=53, scale_lo=118, scale_hi=121)
# Zipf(1) bias: buckets from 1 token to a few hundred (many n-tiles per expert)
ZIPF = si.LayerRecipe("bs_zipf", d=1024, ff=1024, E=24, k=4, T=300, seed=54, bias="zipf", scale_lo=118,
                      scale_hi=121)


@pytest.fixture(scope="module")
def lib():
    from quantized_expert_ffn_score_gb300 import build, moe
    build.build()
    return moe


@pytest.fixture()
def ctx(lib):
    c = lib.Context(0)
    assert c.mxfp4_kernel == "auto"
    c.mxfp4_kernel = "block_scaled"
    yield c
    c.close()


def test_setting_round_trips(lib, ctx):
    for name in ("gemv", "auto"):
        ctx.mxfp4_kernel = name
        assert ctx.mxfp4_kernel == name
    ctx.mxfp4_kernel = "block_scaled"
    assert ctx.mxfp4_kernel == "block_scaled"


def test_small_single_group_padded_ntile(lib, ctx):
    _, counts = gu.full_check(lib, ctx, SMALL)
    assert counts.max() <= 8


def test_split_k_last_arriver(lib, ctx):
    _, counts = gu.full_check(lib, ctx, SPLIT)
    assert counts.sum() == SPLIT.T * SPLIT.k <= 128
    assert 2 * 8 * int((counts > 0).sum()) <= ctx.num_sms  # (d / 128) tiles per expert, two CTAs per tile


def test_split_k_is_deterministic(lib, ctx):
    # two partial sums per split tile, added to a zeroed word: the same bits on every run
    from quantized_expert_ffn_score_gb300 import synthetic
    layer = synthetic.device_layer(SPLIT)
    x = synthetic.device_x(SPLIT)
    outs = [gu.run_layer(lib, ctx, layer, x)[0] for _ in range(3)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_fewer_pairs_than_box_rows(lib, ctx):
    _, counts = gu.full_check(lib, ctx, FEWP)
    assert counts.sum() == 3


def test_mid_ragged_ntiles(lib, ctx):
    _, counts = gu.full_check(lib, ctx, MID)
    assert np.any(counts % 48 != 0) and np.any(counts % 40 != 0)  # ragged gate/up and down n-tiles


def test_zipf_many_ntiles(lib, ctx):
    _, counts = gu.full_check(lib, ctx, ZIPF)
    assert counts.max() > 3 * 48  # several n-tiles for the hottest expert


def test_situ(lib, ctx):
    gu.full_check(lib, ctx, MID.with_(act="situ", seed=55))


def _route(moe, ctx, layer, x, r):
    T = x.shape[0]
    topk = torch.empty((T, r.k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, r.k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(ctx, x, layer.router_w, layer.router_bias, r.k, topk, gates,
                       moe.workspace(moe.route_topk_ws_bytes(T, r.d, r.E, r.k)))
    counts = torch.empty(r.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(r.E + 1, dtype=torch.int32, device="cuda")
    pairs = torch.empty(T * r.k, dtype=torch.int32, device="cuda")
    moe.moe_bucket_tokens(ctx, topk, r.E, counts, offsets, pairs,
                          moe.workspace(moe.bucket_tokens_ws_bytes(T, r.k, r.E)))
    return offsets, pairs


@pytest.mark.parametrize("r", [SPLIT, MID], ids=["split", "mid"])
def test_standalone_expert_call_matches_oracle_pairs(lib, ctx, r):
    from quantized_expert_ffn_score_gb300 import synthetic
    import oracle
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    offsets, pairs = _route(lib, ctx, layer, x, r)
    y = torch.full((r.T * r.k, r.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = lib.workspace(lib.expert_ffn_ws_bytes(r.T, r.k, r.d, r.ff, r.E))
    lib.moe_expert_ffn_mxfp4(ctx, x, r.k, layer, offsets, pairs, y, ws)
    ctx.check()
    y = y.cpu().numpy().astype(np.float64)
    xh = si.layer_x(r)
    _, idx, _ = oracle.router(xh, si.layer_router_w(r), si.layer_bias(r), r.k)
    ref = np.empty_like(y)
    for e in np.unique(idx):
        rec = si.layer_record(r, int(e))
        for p in np.nonzero(idx.reshape(-1) == e)[0]:
            ref[p] = oracle.expert_mxfp4(gu.x_host_f64(xh)[p // r.k], rec, r.d, r.ff, act_kind=r.act)
    gu.assert_rms_close(y, ref, what="block-scaled expert call")


def test_agrees_with_gemv_pair(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = MID
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    outs = []
    for kern in ("block_scaled", "gemv"):
        ctx.mxfp4_kernel = kern
        outs.append(gu.run_layer(lib, ctx, layer, x)[0].astype(np.float64))
    xh = gu.x_host_f64(si.layer_x(r))
    d0, d1 = outs[0] - xh, outs[1] - xh
    rms = np.sqrt(np.mean(d1 ** 2))
    assert np.max(np.abs(d0 - d1)) <= 2 * gu.TOL * rms


def test_missing_expert_is_reported(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = ZIPF
    layer = synthetic.device_layer(r, missing=[0])
    x = synthetic.device_x(r)
    out = torch.empty((r.T, r.d), dtype=torch.float32, device="cuda")
    ws = lib.workspace(lib.layer_forward_ws_bytes(layer, r.T))
    lib.moe_layer_forward(ctx, layer, x, out, ws)
    with pytest.raises(lib.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_MISSING_EXPERT"


def test_k3_decode_one_token(lib, ctx):
    gu.full_check(lib, ctx, si.get_workload("k3_mxfp4_decode_e64"))
