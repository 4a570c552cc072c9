"""Experts beyond HBM (moe_tier_*): a layer whose record table is managed by a
tier -- a heat-ranked set of experts in HBM slots, the others read in place
from page-locked host memory by the same kernels, or absent -- through the C
ABI, against the fp64 oracle.

Cases: part of the bank resident and the rest read from host memory (the
GEMV pair, the block-scaled kernel and the RVQ3 kernels), every expert
resident, a routed expert in no tier reported as missing (never
substituted), and a rebalance after observed routing moving exactly the
hottest experts (the ranking moe_tier_plan fixes) into slots whose bytes then
equal the host records."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

MID = si.LayerRecipe("tier_mid", d=1024, ff=576, E=40, k=6, T=37, seed=81, scale_lo=118, scale_hi=121)
BS = si.LayerRecipe("tier_bs", d=1024, ff=1024, E=24, k=4, T=6, seed=82, scale_lo=118, scale_hi=121)
RVQ = si.LayerRecipe("tier_rvq3", d=1024, ff=576, E=24, k=4, T=11, seed=83, quant="rvq3")


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


def _tiered(moe, ctx, r, n_slots, direct_host=True, decay=1.0):
    """The recipe's layer with its records in page-locked host memory and a
    tier of n_slots HBM slots managing the table the layer reads."""
    from quantized_expert_ffn_score_gb300 import synthetic
    dl = synthetic.device_layer(r)
    n = r.E + r.n_shared
    host = torch.empty(n * dl.stride, dtype=torch.uint8, pin_memory=True)
    host.copy_(dl.bank.cpu())
    slots = torch.empty(max(n_slots, 1) * dl.stride, dtype=torch.uint8, device="cuda")
    table = torch.zeros(n, dtype=torch.int64, device="cuda")
    tier = moe.Tier(ctx, n, si.record_size(r), dl.stride, host, slots, n_slots, table, direct_host=direct_host,
                    decay=decay)
    layer = moe.Layer(r.d, r.ff, r.E, r.k, dl.router_w, table, quant=r.quant, act=r.act,
                      router_bias=dl.router_bias, codebooks=dl.codebooks, keep=[host, slots], n_shared=r.n_shared,
                      bias_mode=r.bias_mode)
    layer.recipe = r
    del dl  # the full device bank is no longer needed
    torch.cuda.empty_cache()
    return layer, tier, host, slots


def _check_layer(moe, ctx, layer, r, name):
    from quantized_expert_ffn_score_gb300 import synthetic
    x = synthetic.device_x(r)
    out, topk, gates, counts = gu.run_layer(moe, ctx, layer, x)
    xh = si.layer_x(r)
    logits, idx, g, y, _ = gu.oracle_layer(r, xh)
    gu.check_routing(topk[:, :r.k], gates[:, :r.k], idx, g, gu.gate_tolerance(r, xh, logits))
    delta = out.astype(np.float64) - gu.x_host_f64(xh)
    err, rms = gu.rms_err(delta, y)
    gu.record_margin(name, err, rms, r.T)
    gu.assert_rms_close(delta, y, what=name)
    return counts


def test_quarter_resident_rest_read_from_host_memory(lib, ctx):
    r = MID
    layer, tier, host, slots = _tiered(lib, ctx, r, n_slots=10)
    tier.pin(list(range(0, 40, 4)))  # every fourth expert in HBM
    slot, _ = tier.residency()
    assert sorted(np.nonzero(slot >= 0)[0].tolist()) == list(range(0, 40, 4))
    counts = _check_layer(lib, ctx, layer, r, "tier_mid_quarter")
    used = np.nonzero(counts > 0)[0]
    assert np.any(slot[used] >= 0) and np.any(slot[used] < 0), "needs resident and host-read experts in one call"
    tier.close()


def test_all_resident(lib, ctx):
    r = MID
    layer, tier, _, _ = _tiered(lib, ctx, r, n_slots=r.E)
    tier.pin(list(range(r.E)))
    _check_layer(lib, ctx, layer, r, "tier_mid_all")
    tier.close()


def test_expert_in_no_tier_is_missing(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = MID
    layer, tier, _, _ = _tiered(lib, ctx, r, n_slots=10, direct_host=False)
    tier.pin(list(range(10)))
    x = synthetic.device_x(r)
    out = torch.empty((r.T, r.d), dtype=torch.float32, device="cuda")
    lib.moe_layer_forward(ctx, layer, x, out, lib.workspace(lib.layer_forward_ws_bytes(layer, r.T)))
    with pytest.raises(lib.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_MISSING_EXPERT" and ei.value.detail >= 10
    tier.close()


def test_rebalance_moves_the_hottest_experts_in(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = MID
    n_slots = 8
    layer, tier, host, slots = _tiered(lib, ctx, r, n_slots=n_slots)
    counts = torch.empty(r.E, dtype=torch.int32, device="cuda")
    out = torch.empty((r.T, r.d), dtype=torch.float32, device="cuda")
    ws = lib.workspace(lib.layer_forward_ws_bytes(layer, r.T))
    heat = np.zeros(r.E)
    cur = np.full(r.E, -1, dtype=np.int32)
    for step, off in enumerate((0, 200, 400)):
        x = synthetic.device_x(r, token_offset=off)
        lib.moe_layer_forward(ctx, layer, x, out, ws, counts_out=counts)
        ctx.check()
        tier.observe(counts)
        heat += counts.cpu().numpy()
        moved = tier.rebalance()
        torch.cuda.synchronize()
        want, n_want = lib.tier_plan(heat, np.ones(r.E), cur, n_slots)
        slot, h = tier.residency()
        np.testing.assert_array_equal(slot, want)
        np.testing.assert_allclose(h, heat)
        assert moved == n_want
        cur = slot
        # the slots hold the host records byte for byte
        nb = si.record_size(r)
        stride = host.numel() // r.E
        hb = host.numpy()
        sb = slots.cpu().numpy()
        for e in np.nonzero(slot >= 0)[0]:
            s = int(slot[e])
            np.testing.assert_array_equal(sb[s * stride:s * stride + nb], hb[e * stride:e * stride + nb])
    _check_layer(lib, ctx, layer, r, "tier_mid_rebalanced")
    tier.close()


def test_block_scaled_kernel_reads_host_records(lib, ctx):
    r = BS
    layer, tier, _, _ = _tiered(lib, ctx, r, n_slots=6)
    tier.pin([0, 3, 5, 7, 11, 13])
    assert ctx.mxfp4_kernel == "auto"  # 6 tokens, 512-multiple shapes: the block-scaled kernel
    _check_layer(lib, ctx, layer, r, "tier_bs_quarter")
    tier.close()


def test_rvq3_half_resident(lib, ctx):
    r = RVQ
    layer, tier, _, _ = _tiered(lib, ctx, r, n_slots=12)
    tier.pin(list(range(0, 24, 2)))
    _check_layer(lib, ctx, layer, r, "tier_rvq3_half")
    tier.close()


def test_invalid_descriptions_are_refused(lib, ctx):
    r = MID
    nb = si.record_size(r)
    stride = (nb + 4095) // 4096 * 4096
    host = torch.empty(4 * stride, dtype=torch.uint8, pin_memory=True)
    slots = torch.empty(2 * stride, dtype=torch.uint8, device="cuda")
    table = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(lib.MoeError):  # more slots than experts
        lib.Tier(ctx, 4, nb, stride, host, slots, 5, table)
    with pytest.raises(lib.MoeError):  # stride not a multiple of 256
        lib.Tier(ctx, 4, nb, stride + 16, host, slots, 2, table)
    with pytest.raises(lib.MoeError):  # decay out of range
        lib.Tier(ctx, 4, nb, stride, host, slots, 2, table, decay=0.0)
    pageable = torch.empty(4 * stride, dtype=torch.uint8)  # not page-locked
    with pytest.raises(lib.MoeError):
        lib.Tier(ctx, 4, nb, stride, pageable, slots, 2, table)
    t = lib.Tier(ctx, 4, nb, stride, host, slots, 2, table)
    with pytest.raises(lib.MoeError):
        t.pin([0, 1, 2])  # more than the slots
    t.close()


@pytest.mark.slow
def test_k3_decode_quarter_resident(lib, ctx):
    r = si.get_workload("k3_mxfp4_decode").with_(name="k3_mxfp4_decode_tier25")
    layer, tier, _, _ = _tiered(lib, ctx, r, n_slots=r.E // 4)
    tier.pin(list(range(0, r.E, 4)))
    _check_layer(lib, ctx, layer, r, r.name)
    tier.close()
