"""moe_expert_ffn_mxfp4_static: the expert FFN for callers that cannot allocate
device memory (the scratch is a static array inside the library instead of a
caller workspace).  Called through the C ABI twice in a row, on different
tokens, its outputs must match moe_expert_ffn_mxfp4's within the parity
tolerance; at shapes where the workspace call takes the block-scaled kernel
(the static call always runs the GEMV pair) both are held to the oracle; a
call whose scratch would not fit is refused.

This file is collected last so that a stop-at-first-failure run has run every
other test before it; it builds everything it needs itself, so it also passes
alone in a fresh process."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

RECIPE = si.LayerRecipe("no_alloc", d=1024, ff=576, E=40, k=6, T=37, seed=31, scale_lo=118, scale_hi=121)


@pytest.fixture(scope="module")
def env():
    from quantized_expert_ffn_score_gb300 import build, moe, synthetic
    build.build()
    ctx = moe.Context(0)
    layer = synthetic.device_layer(RECIPE)
    yield moe, synthetic, ctx, layer
    ctx.close()


def _route(moe, ctx, layer, x):
    r = RECIPE
    T = x.shape[0]
    topk = torch.empty((T, r.k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, r.k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(ctx, x, layer.router_w, None, r.k, topk, gates, moe.workspace(moe.route_topk_ws_bytes(T, r.d,
                                                                                                              r.E, r.k)))
    counts = torch.empty(r.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(r.E + 1, dtype=torch.int32, device="cuda")
    pairs = torch.empty(T * r.k, dtype=torch.int32, device="cuda")
    moe.moe_bucket_tokens(ctx, topk, r.E, counts, offsets, pairs, moe.workspace(moe.bucket_tokens_ws_bytes(T, r.k,
                                                                                                          r.E)))
    return offsets, pairs


def test_static_scratch_matches_workspace_path_twice(env):
    moe, synthetic, ctx, layer = env
    r = RECIPE
    for call, offset in enumerate((0, 100)):  # two calls in a row, different tokens
        x = synthetic.device_x(r, token_offset=offset)
        offsets, pairs = _route(moe, ctx, layer, x)
        y_ws = torch.empty((r.T * r.k, r.d), dtype=torch.float32, device="cuda")
        ws = moe.workspace(moe.expert_ffn_ws_bytes(r.T, r.k, r.d, r.ff, r.E))
        moe.moe_expert_ffn_mxfp4(ctx, x, r.k, layer, offsets, pairs, y_ws, ws)
        y_static = torch.full((r.T * r.k, r.d), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_expert_ffn_mxfp4_static(ctx, x, r.k, layer, offsets, pairs, y_static)
        ctx.check()
        ref = y_ws.cpu().numpy().astype(np.float64)
        got = y_static.cpu().numpy().astype(np.float64)
        gu.assert_rms_close(got, ref, what=f"static-scratch call {call + 1}")


# d and ff multiples of 512 and several tokens: the workspace call takes the
# block-scaled tensor-core kernel here, while the static call always runs the
# GEMV pair, so the two differ in rounding and both are held to the oracle.
RECIPE_512 = si.LayerRecipe("no_alloc_512", d=1024, ff=1024, E=16, k=4, T=6, seed=32, scale_lo=118, scale_hi=121)


def test_static_scratch_at_block_scaled_shapes_matches_oracle_twice(env):
    import oracle
    moe, synthetic, ctx, _ = env
    r = RECIPE_512
    layer = synthetic.device_layer(r)
    assert ctx.mxfp4_kernel == "auto"
    for call, offset in enumerate((0, 50)):
        x = synthetic.device_x(r, token_offset=offset)
        T = x.shape[0]
        topk = torch.empty((T, r.k), dtype=torch.int32, device="cuda")
        gates = torch.empty((T, r.k), dtype=torch.float32, device="cuda")
        moe.moe_route_topk(ctx, x, layer.router_w, None, r.k, topk, gates,
                           moe.workspace(moe.route_topk_ws_bytes(T, r.d, r.E, r.k)))
        counts = torch.empty(r.E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(r.E + 1, dtype=torch.int32, device="cuda")
        pairs = torch.empty(T * r.k, dtype=torch.int32, device="cuda")
        moe.moe_bucket_tokens(ctx, topk, r.E, counts, offsets, pairs,
                              moe.workspace(moe.bucket_tokens_ws_bytes(T, r.k, r.E)))
        y_ws = torch.empty((T * r.k, r.d), dtype=torch.float32, device="cuda")
        moe.moe_expert_ffn_mxfp4(ctx, x, r.k, layer, offsets, pairs, y_ws,
                                 moe.workspace(moe.expert_ffn_ws_bytes(T, r.k, r.d, r.ff, r.E)))
        y_static = torch.full((T * r.k, r.d), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_expert_ffn_mxfp4_static(ctx, x, r.k, layer, offsets, pairs, y_static)
        ctx.check()
        # the oracle's per-pair outputs y_pairs[p] = expert(topk[p]) applied to x[p // k]
        idx = topk.cpu().numpy().reshape(-1)
        xh = gu.x_host_f64(si.layer_x(r, T=T, token_offset=offset))
        ref = np.empty((T * r.k, r.d))
        for e in np.unique(idx):
            rec = si.layer_record(r, int(e))
            for p in np.nonzero(idx == e)[0]:
                ref[p] = oracle.expert_mxfp4(xh[p // r.k], rec, r.d, r.ff, act_kind=r.act)
        gu.assert_rms_close(y_static.cpu().numpy().astype(np.float64), ref, what=f"static call {call + 1}")
        gu.assert_rms_close(y_ws.cpu().numpy().astype(np.float64), ref, what=f"workspace call {call + 1}")


def test_static_scratch_refuses_oversized_calls(env):
    moe, synthetic, ctx, layer = env
    r = RECIPE
    T = moe.expert_ffn_static_max_bytes() // (r.k * r.ff * 4) + 1  # h alone would exceed the array
    x = torch.zeros((T, r.d), dtype=torch.bfloat16, device="cuda")
    offsets = torch.zeros(r.E + 1, dtype=torch.int32, device="cuda")
    pairs = torch.zeros(T * r.k, dtype=torch.int32, device="cuda")
    y = torch.empty((T * r.k, r.d), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_expert_ffn_mxfp4_static(ctx, x, r.k, layer, offsets, pairs, y)
    assert ei.value.name == "MOE_ERR_UNSUPPORTED"
    ctx.check()
