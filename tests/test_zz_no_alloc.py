"""moe_expert_ffn_mxfp4_static: the expert FFN for callers that cannot allocate
device memory (the scratch is a static array inside the library instead of a
caller workspace).  Called through the C ABI twice in a row, on different
tokens, its outputs must match moe_expert_ffn_mxfp4's within the parity
tolerance; a call whose scratch would not fit is refused.

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
