"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Routing indices and bucket contents must be identical;
outputs within 2e-3 x RMS of the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from quantized_expert_ffn_score_gb300 import build, moe
    build.build()
    return moe


@pytest.fixture(scope="module")
def ctx(lib):
    c = lib.Context(0)
    yield c
    c.close()


MID_MX = si.LayerRecipe("mid_mxfp4", d=1024, ff=576, E=40, k=6, T=37, seed=11, scale_lo=118, scale_hi=121)
MID_RVQ = si.LayerRecipe("mid_rvq3", d=1024, ff=576, E=24, k=4, T=11, seed=12, quant="rvq3")


def test_tiny_layer(lib, ctx):
    gu.full_check(lib, ctx, si.get_workload("tiny"))


def test_mid_mxfp4_spans_tiles_and_ragged_tail(lib, ctx):
    gu.full_check(lib, ctx, MID_MX)


def test_mid_mxfp4_situ_fp32_router(lib, ctx):
    gu.full_check(lib, ctx, MID_MX.with_(act="situ", x_dtype="f32", w_dtype="f32", seed=13))


def test_mid_mxfp4_bf16_x_fp32_router(lib, ctx):
    gu.full_check(lib, ctx, MID_MX.with_(w_dtype="f32", seed=14, T=5, k=1))


def test_mid_mxfp4_odd_expert_count_tiled_router(lib, ctx):
    # 37 experts (the last expert-row pair of a warp has one row) and 29 tokens
    # (a ragged last tile of 8 and a ragged second pass of 4)
    gu.full_check(lib, ctx, MID_MX.with_(E=37, k=5, T=29, seed=17))


def test_mid_mxfp4_all_experts_selected(lib, ctx):
    gu.full_check(lib, ctx, MID_MX.with_(E=8, k=8, T=3, seed=15))


@pytest.mark.parametrize("quant", ["mxfp4", "rvq3"])
def test_one_token_layer_without_optional_outputs(lib, ctx, quant):
    # one token with no routing outputs asked for: the top-k kernel buckets the
    # pairs and writes no per-expert counts; the output must still match the oracle
    moe = lib
    from quantized_expert_ffn_score_gb300 import synthetic
    r = (MID_MX if quant == "mxfp4" else MID_RVQ).with_(T=1, seed=33)
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    out = torch.empty((1, r.d), dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.layer_forward_ws_bytes(layer, 1))
    moe.moe_layer_forward(ctx, layer, x, out, ws)
    ctx.check()
    xh = si.layer_x(r)
    _, _, _, y, _ = gu.oracle_layer(r, xh)
    delta = out.cpu().numpy().astype(np.float64) - gu.x_host_f64(xh)
    gu.assert_rms_close(delta, y, what=f"one token, {quant}, no optional outputs")


def test_mid_rvq3(lib, ctx):
    gu.full_check(lib, ctx, MID_RVQ)


def test_mid_rvq3_situ(lib, ctx):
    gu.full_check(lib, ctx, MID_RVQ.with_(act="situ", seed=16, T=3))


# Two shared experts after the routed ones and the score-correction bias
# steering the selection only (the K3 MoE block's routing).
SHARED_MX = MID_MX.with_(n_shared=2, bias="zipf", bias_mode="select", seed=21)


@pytest.mark.parametrize("T", [1, 5, 37])
def test_mid_mxfp4_shared_experts_select_bias(lib, ctx, T):
    # one token: the top-k kernel buckets the 6 + 2 pairs itself and the GEMV
    # runs them; 5 tokens: compensated router, block-scaled experts; 37 tokens:
    # tiled router, shared experts with 37 tokens each
    gu.full_check(lib, ctx, SHARED_MX.with_(T=T))


def test_mid_mxfp4_shared_expert_additive_bias_fp32(lib, ctx):
    # fp32 x and router: the FMA GEMV and the fp32 router kernels
    gu.full_check(lib, ctx, MID_MX.with_(n_shared=1, bias="zipf", x_dtype="f32", w_dtype="f32", T=3, seed=22))


def test_mid_mxfp4_select_bias_without_shared_experts(lib, ctx):
    gu.full_check(lib, ctx, MID_MX.with_(bias="zipf", bias_mode="select", T=23, seed=24))


def test_mid_rvq3_shared_experts(lib, ctx):
    gu.full_check(lib, ctx, MID_RVQ.with_(n_shared=2, bias="zipf", bias_mode="select", seed=23))


@pytest.mark.slow
def test_k3_mxfp4_decode_shared2(lib, ctx):
    gu.full_check(lib, ctx, si.get_workload("k3_mxfp4_decode_shared2"))


@pytest.mark.slow
def test_k3_mxfp4_prefill_shared2_e64(lib, ctx):
    # 40 tokens over 64 experts plus the 2 shared ones (40 tokens each): every
    # token's routing, counts and output
    gu.full_check(lib, ctx, si.get_workload("k3_mxfp4_prefill_shared2_e64"))


@pytest.mark.slow
def test_k3_mxfp4_decode_b1(lib, ctx):
    gu.full_check(lib, ctx, si.get_workload("k3_mxfp4_decode"))


@pytest.mark.slow
def test_k3_rvq3_decode_b1(lib, ctx):
    gu.full_check(lib, ctx, si.get_workload("k3_rvq3_decode_b1"))


@pytest.mark.slow
def test_k3_rvq3_decode_b8(lib, ctx):
    gu.full_check(lib, ctx, si.get_workload("k3_rvq3_decode_b8"))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["k3_mxfp4_prefill_zipf", "k3_mxfp4_prefill_uniform"])
def test_k3_prefill_all_tokens(lib, ctx, name):
    # 512 tokens, 8,192 pairs: every token's routing, counts and output against
    # the oracle (Zipf: hot buckets of hundreds of tokens in several 48/40-token
    # n-tiles with ragged tails; uniform: ~9 tokens on each of ~896 experts)
    _, counts = gu.full_check(lib, ctx, si.get_workload(name))
    if name.endswith("zipf"):
        assert counts.max() > 3 * 48 and np.any((counts > 48) & (counts % 48 != 0))


def test_route_topk_and_bucket_standalone_match_oracle(lib, ctx):
    # the K3 router on 512 tokens, with and without the Zipf bias, then bucketing
    moe = lib
    from quantized_expert_ffn_score_gb300 import synthetic
    for name in ("k3_mxfp4_prefill_zipf", "k3_mxfp4_prefill_uniform"):
        r = si.get_workload(name)
        W = torch.empty((r.E, r.d), dtype=torch.bfloat16, device="cuda")
        si.dev_layer_router_w(r, W.data_ptr())
        b = si.layer_bias(r)
        bias = None if b is None else torch.from_numpy(b).cuda()
        x = synthetic.device_x(r)
        topk = torch.empty((r.T, r.k), dtype=torch.int32, device="cuda")
        gates = torch.empty((r.T, r.k), dtype=torch.float32, device="cuda")
        ws = moe.workspace(moe.route_topk_ws_bytes(r.T, r.d, r.E, r.k))
        moe.moe_route_topk(ctx, x, W, bias, r.k, topk, gates, ws)
        counts = torch.empty(r.E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(r.E + 1, dtype=torch.int32, device="cuda")
        pairs = torch.empty(r.T * r.k, dtype=torch.int32, device="cuda")
        wsb = moe.workspace(moe.bucket_tokens_ws_bytes(r.T, r.k, r.E))
        moe.moe_bucket_tokens(ctx, topk, r.E, counts, offsets, pairs, wsb)
        ctx.check()
        xh = si.layer_x(r)
        logits, idx, g = oracle.router(xh, si.layer_router_w(r), b, r.k)
        gu.check_routing(topk.cpu().numpy(), gates.cpu().numpy(), idx, g, gu.gate_tolerance(r, xh, logits))
        c_ref, o_ref, p_ref = oracle.bucket(idx, r.E)
        np.testing.assert_array_equal(counts.cpu().numpy(), c_ref)
        np.testing.assert_array_equal(offsets.cpu().numpy(), o_ref)
        np.testing.assert_array_equal(pairs.cpu().numpy(), p_ref)


@pytest.mark.parametrize("E,k,T", [(1536, 8, 5), (100, 32, 7), (1024, 31, 3)])
def test_route_topk_radix_and_warp_select_paths(lib, ctx, E, k, T):
    # E > 1024 or k + 1 > 32 take the radix select; E <= 1024 with k + 1 <= 32
    # the warp select (the last case sits at both limits)
    moe = lib
    d = 256
    rng = np.random.default_rng(E + k)
    Wb = torch.from_numpy((rng.standard_normal((E, d)) / 16).astype(np.float32)).to(torch.bfloat16)
    x = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    topk = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.route_topk_ws_bytes(T, d, E, k))
    moe.moe_route_topk(ctx, x.cuda(), Wb.cuda(), None, k, topk, gates, ws)
    ctx.check()
    xh = x.view(torch.int16).numpy().view(np.uint16)
    Wh = Wb.view(torch.int16).numpy().view(np.uint16)
    logits, idx, g = oracle.router(xh, Wh, None, k)
    # logits are O(1) here, so the fp32 logit and gate roundings move a gate by
    # a few 1e-7 relative; 2e-5 leaves ample room
    gu.check_routing(topk.cpu().numpy(), gates.cpu().numpy(), idx, g, np.full(T, 2e-5))


@pytest.mark.parametrize("T", [8, 512])
def test_route_topk_ex_select_bias_matches_oracle(lib, ctx, T):
    # the K3 router with the Zipf bias for the selection only: 8 tokens
    # (compensated sums) and 512 (tiled); the selection equals the additive
    # mode's (the keys are the same), the gates come from the unbiased logits
    moe = lib
    from quantized_expert_ffn_score_gb300 import synthetic
    r = si.get_workload("k3_mxfp4_prefill_zipf").with_(T=T, bias_mode="select")
    W = torch.empty((r.E, r.d), dtype=torch.bfloat16, device="cuda")
    si.dev_layer_router_w(r, W.data_ptr())
    b = si.layer_bias(r)
    bias = torch.from_numpy(b).cuda()
    x = synthetic.device_x(r)
    topk = torch.empty((T, r.k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, r.k), dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.route_topk_ws_bytes(T, r.d, r.E, r.k))
    moe.moe_route_topk_ex(ctx, x, W, bias, "select", r.k, topk, gates, ws)
    topk_add = torch.empty_like(topk)
    gates_add = torch.empty_like(gates)
    moe.moe_route_topk(ctx, x, W, bias, r.k, topk_add, gates_add, ws)
    ctx.check()
    xh = si.layer_x(r)
    logits, idx, g = oracle.router(xh, si.layer_router_w(r), b, r.k, bias_mode="select")
    gu.check_routing(topk.cpu().numpy(), gates.cpu().numpy(), idx, g, gu.gate_tolerance(r, xh, logits))
    np.testing.assert_array_equal(topk_add.cpu().numpy(), idx)
    assert not np.allclose(gates_add.cpu().numpy(), gates.cpu().numpy(), rtol=1e-3)


@pytest.mark.parametrize("T", [3, 20])
def test_route_topk_ex_forced_selection_gates_ignore_the_bias(lib, ctx, T):
    # a bias of about 1000 on k chosen experts makes them the selection; their
    # gates are the softmax of the logits without the bias, which the bias's
    # own fp32 rounding (about 6e-5 at 1000) must not reach
    moe = lib
    E, d, k = 256, 512, 8
    rng = np.random.default_rng(T)
    Wb = torch.from_numpy((rng.standard_normal((E, d)) / 16).astype(np.float32)).to(torch.bfloat16)
    x = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    chosen = rng.choice(E, size=k, replace=False)
    b = np.zeros(E, dtype=np.float32)
    b[chosen] = 1000.0 - 10.0 * np.arange(k, dtype=np.float32)
    topk = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.route_topk_ws_bytes(T, d, E, k))
    moe.moe_route_topk_ex(ctx, x.cuda(), Wb.cuda(), torch.from_numpy(b).cuda(), "select", k, topk, gates, ws)
    ctx.check()
    xh = x.view(torch.int16).numpy().view(np.uint16)
    Wh = Wb.view(torch.int16).numpy().view(np.uint16)
    logits, idx, g = oracle.router(xh, Wh, b, k, bias_mode="select")
    assert np.all(idx == chosen[None, :])
    gu.check_routing(topk.cpu().numpy(), gates.cpu().numpy(), idx, g, np.full(T, 2e-5))


@pytest.mark.parametrize("T", [16, 300])
def test_router_certifies_exact_ties_and_near_ties(lib, ctx, T):
    # duplicated router rows give exactly equal logits (ties must go to the lower
    # index); rows differing in one low bit give near-ties the fp32 bound cannot
    # separate, forcing the fp64 and sequential-fp64 recomputation paths.  16
    # tokens: compensated logits, one top-k CTA per SM; 300 tokens (more than
    # the SMs): the tiled fp32 logits and the top-k launched 4 CTAs per SM
    moe = lib
    d, E, k = 256, 64, 8
    rng = np.random.default_rng(0)
    Wf = (rng.standard_normal((E, d)) / 16).astype(np.float32)
    Wb = torch.from_numpy(Wf).to(torch.bfloat16)
    Wb[10] = Wb[3]
    Wb[40] = Wb[3]
    Wb[20] = Wb[7]
    w16 = Wb.view(torch.int16)
    w16[21] = w16[7]
    w16[21, 5] += 1  # one ulp apart in one weight
    x = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    x[:, :] = x[0]  # every token the same: the tied experts appear in many top-k sets
    x[1:, 0] += torch.arange(1, T, dtype=torch.bfloat16) * 0.01
    Wd, xd = Wb.cuda(), x.cuda()
    topk = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.route_topk_ws_bytes(T, d, E, k))
    ctx.stats()
    moe.moe_route_topk(ctx, xd, Wd, None, k, topk, gates, ws)
    ctx.check()
    fp64_tokens, seq_logits = ctx.stats()
    assert fp64_tokens > 0 and seq_logits > 0  # both recheck passes ran
    xh = x.view(torch.int16).numpy().view(np.uint16)
    Wh = Wb.view(torch.int16).numpy().view(np.uint16)
    logits, idx, g = oracle.router(xh, Wh, None, k)
    np.testing.assert_array_equal(topk.cpu().numpy(), idx)


def test_stack_layers_individually_and_chained(lib, ctx):
    """Six K3-shaped... reduced to a mid shape here; the full-size stack is in
    test_k3_stack.  Each layer on its own seeded input, then the chain."""
    moe = lib
    from quantized_expert_ffn_score_gb300 import synthetic
    recipes = [MID_MX.with_(seed=200 + l, T=9) for l in range(3)]
    layers = [synthetic.device_layer(r) for r in recipes]
    x0 = synthetic.device_x(recipes[0])
    out = torch.empty((9, MID_MX.d), dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.stack_forward_ws_bytes(layers, 9))
    moe.moe_stack_forward(ctx, layers, x0, out, ws)
    ctx.check()
    # the chain by hand through moe_layer_forward must give the same bits
    x = x0
    for i, (r, layer) in enumerate(zip(recipes, layers)):
        last = i == len(recipes) - 1
        o = torch.empty((9, r.d), dtype=torch.float32 if last else torch.bfloat16, device="cuda")
        w = moe.workspace(moe.layer_forward_ws_bytes(layer, 9))
        moe.moe_layer_forward(ctx, layer, x, o, w)
        x = o
    ctx.check()
    assert torch.equal(x, out)


def test_combine_bf16_output_rounds_fp32_sum(lib, ctx):
    moe = lib
    T, k, d = 5, 3, 64
    g = torch.rand((T, k), device="cuda")
    g[2, 1] = 0.0
    y = torch.randn((T * k, d), device="cuda")
    y[2 * k + 1] = float("nan")  # gate 0: never read
    xr = torch.randn((T, d), device="cuda").to(torch.bfloat16)
    out32 = torch.empty((T, d), device="cuda")
    out16 = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(ctx, xr, y, g, k, out32)
    moe.moe_combine(ctx, xr, y, g, k, out16)
    ctx.check()
    assert torch.isfinite(out32).all()
    assert torch.equal(out32.to(torch.bfloat16), out16)
    ref = oracle.combine(xr.float().cpu().numpy().astype(np.float64), torch.nan_to_num(y).cpu().double().numpy(),
                         g.cpu().double().numpy(), k)
    np.testing.assert_allclose(out32.cpu().numpy(), ref, rtol=1e-5, atol=1e-5)
