"""The tensor-core path of the MXFP4 expert FFN (grouped GEMM for experts with
many tokens) against the fp64 oracle, through the C ABI.

The path is chosen per expert by its token count (moe_ctx_set_gemm_min_tokens):
these cases run it beside the GEMV path (a Zipf-skewed router: a few experts
with several 128-token blocks and ragged tails, many with a handful), alone
(threshold 1: every expert, down to one token, on the tensor cores), with the
last bucket of the slot range hot (its final token box reaches past the end of
the activations), with SiTU, through the standalone expert call, and with a
hot expert's record missing.  The context selects that kernel pair
(moe_ctx_set_mxfp4_kernel); the block-scaled kernel has its own tests."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

# d, ff multiples of 256 (the GEMM path's tiling); Zipf(1) bias over 24 experts
ZIPF = si.LayerRecipe("gemm_zipf", d=512, ff=512, E=24, k=4, T=300, seed=41, bias="zipf", scale_lo=118, scale_hi=121)
# 8 experts, 2 of them per token: every bucket ~50 tokens, the last one hot too
UNIFORM = si.LayerRecipe("gemm_uniform", d=256, ff=256, E=8, k=2, T=203, seed=42)


@pytest.fixture(scope="module")
def lib():
    from quantized_expert_ffn_score_gb300 import build, moe
    build.build()
    return moe


@pytest.fixture()
def ctx(lib):
    c = lib.Context(0)
    c.mxfp4_kernel = "gemv_gemm"  # these cases are about that kernel pair
    yield c
    c.close()


def test_default_threshold(lib, ctx):
    assert ctx.gemm_min_tokens == 2
    with pytest.raises(lib.MoeError):
        ctx.gemm_min_tokens = -1


def test_gemm_and_gemv_experts_in_one_layer(lib, ctx):
    ctx.gemm_min_tokens = 8
    _, counts = gu.full_check(lib, ctx, ZIPF)
    assert counts.max() > 2 * 128, "needs an expert with several token blocks"
    assert np.any((counts > 0) & (counts < 8)), "needs experts on the GEMV path too"
    assert np.any((counts >= 8) & (counts % 16 != 0)), "needs a ragged token tail"


def test_every_expert_on_tensor_cores(lib, ctx):
    ctx.gemm_min_tokens = 1
    _, counts = gu.full_check(lib, ctx, ZIPF.with_(seed=44, T=200))
    assert np.any(counts == 1) and counts.max() > 128


def test_last_bucket_hot_reaches_end_of_slots(lib, ctx):
    ctx.gemm_min_tokens = 1
    _, counts = gu.full_check(lib, ctx, UNIFORM)
    assert counts[-1] > 0 and counts[-1] % 16 != 0


def test_gemm_path_situ(lib, ctx):
    ctx.gemm_min_tokens = 1
    gu.full_check(lib, ctx, ZIPF.with_(act="situ", seed=43))


def test_gemm_path_off_matches_oracle_too(lib, ctx):
    ctx.gemm_min_tokens = 0
    gu.full_check(lib, ctx, ZIPF)


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


def test_standalone_expert_call_both_paths(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = ZIPF
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    offsets, pairs = _route(lib, ctx, layer, x, r)
    ys = []
    for gmin in (0, 1, 8):
        ctx.gemm_min_tokens = gmin
        y = torch.full((r.T * r.k, r.d), float("nan"), dtype=torch.float32, device="cuda")
        ws = lib.workspace(lib.expert_ffn_ws_bytes(r.T, r.k, r.d, r.ff, r.E))
        lib.moe_expert_ffn_mxfp4(ctx, x, r.k, layer, offsets, pairs, y, ws)
        ctx.check()
        ys.append(y.cpu().numpy().astype(np.float64))
    # the oracle's per-pair outputs (ungated): y_pairs[p] = expert(topk[p]) applied to x[p // k]
    import oracle
    xh = si.layer_x(r)
    _, idx, _ = oracle.router(xh, si.layer_router_w(r), si.layer_bias(r), r.k)
    ref = np.empty_like(ys[0])
    for e in np.unique(idx):
        rec = si.layer_record(r, int(e))
        for p in np.nonzero(idx.reshape(-1) == e)[0]:
            ref[p] = oracle.expert_mxfp4(gu.x_host_f64(xh)[p // r.k], rec, r.d, r.ff, act_kind=r.act)
    for gmin, y in zip((0, 1, 8), ys):
        gu.assert_rms_close(y, ref, what=f"expert call, gemm_min_tokens={gmin}")


def test_missing_hot_expert_is_reported(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = ZIPF
    layer = synthetic.device_layer(r, missing=[0])  # expert 0 has the largest bucket under the Zipf bias
    x = synthetic.device_x(r)
    out = torch.empty((r.T, r.d), dtype=torch.float32, device="cuda")
    ws = lib.workspace(lib.layer_forward_ws_bytes(layer, r.T))
    lib.moe_layer_forward(ctx, layer, x, out, ws)
    with pytest.raises(lib.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_MISSING_EXPERT"
