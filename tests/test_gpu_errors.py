"""Device-detected errors and host validation through the C ABI, and the
device generator against the host generator.  Nothing here faults a GPU: a
missing expert is a NULL entry the kernel checks, a bad expert index is a value
the bucketing kernel range-checks."""
import time

import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import gpu_util as gu

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


def test_device_generator_matches_host():
    r = si.get_workload("tiny")
    from quantized_expert_ffn_score_gb300 import synthetic
    layer = synthetic.device_layer(r)
    torch.cuda.synchronize()
    bank = layer.bank.cpu().numpy()
    for e in (0, 7, 15):
        ref = si.layer_record(r, e)
        np.testing.assert_array_equal(bank[e * layer.stride:e * layer.stride + ref.size], ref)
    np.testing.assert_array_equal(layer.router_w.view(torch.int32).cpu().numpy().view(np.float32),
                                  si.layer_router_w(r))
    x = synthetic.device_x(r, T=3, token_offset=2)
    np.testing.assert_array_equal(x.cpu().numpy(), si.layer_x(r, T=3, token_offset=2))
    rv = si.get_workload("k3_rvq3_decode_b1").with_(d=256, ff=128, E=4)
    lv = synthetic.device_layer(rv)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(lv.codebooks[0].cpu().numpy().view(np.uint16).reshape(3, 256, 8),
                                  si.layer_codebooks(rv))
    b = lv.bank.cpu().numpy()
    np.testing.assert_array_equal(b[lv.stride:lv.stride + si.rvq3_record_size(256, 128)], si.layer_record(rv, 1))
    xb = synthetic.device_x(si.get_workload("k3_mxfp4_decode"), T=2)
    np.testing.assert_array_equal(xb.view(torch.int16).cpu().numpy().view(np.uint16),
                                  si.layer_x(si.get_workload("k3_mxfp4_decode"), T=2))


def test_missing_routed_expert_is_reported(moe, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = si.get_workload("tiny")
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    out = torch.empty((r.T, r.d), device="cuda")
    topk = torch.empty((r.T, r.k), dtype=torch.int32, device="cuda")
    ws = moe.workspace(moe.layer_forward_ws_bytes(layer, r.T))
    moe.moe_layer_forward(ctx, layer, x, out, ws, topk_idx_out=topk)
    ctx.check()
    victim = int(topk[0, 0])
    broken = synthetic.device_layer(r, missing=[victim])
    moe.moe_layer_forward(ctx, broken, x, out, ws)
    with pytest.raises(moe.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_MISSING_EXPERT" and ei.value.detail == victim
    ctx.check()  # the error word was cleared and the context still works
    moe.moe_layer_forward(ctx, layer, x, out, ws)
    ctx.check()


def test_missing_shared_expert_is_reported(moe, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = si.get_workload("tiny").with_(n_shared=2)
    x = synthetic.device_x(r)
    out = torch.empty((r.T, r.d), device="cuda")
    broken = synthetic.device_layer(r, missing=[r.E + 1])
    ws = moe.workspace(moe.layer_forward_ws_bytes(broken, r.T))
    moe.moe_layer_forward(ctx, broken, x, out, ws)
    with pytest.raises(moe.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_MISSING_EXPERT" and ei.value.detail == r.E + 1
    ctx.check()


def test_layer_shared_expert_and_bias_mode_validation(moe, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = si.get_workload("tiny").with_(n_shared=2)
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    out = torch.empty((r.T, r.d), device="cuda")
    ws = moe.workspace(moe.layer_forward_ws_bytes(layer, r.T))
    s = layer.struct
    s.bias_mode = 7
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(ctx, layer, x, out, ws)
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    s.bias_mode = 1
    s.mxfp4.E = r.E  # the bank must hold the routed and the shared records
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(ctx, layer, x, out, ws)
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    s.mxfp4.E = r.E + r.n_shared
    s.n_shared = 32 - r.k + 1  # k + n_shared above 32
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(ctx, layer, x, out, ws)
    assert ei.value.name == "MOE_ERR_UNSUPPORTED"
    s.n_shared = r.n_shared
    s.bias_mode = 0
    moe.moe_layer_forward(ctx, layer, x, out, ws)
    ctx.check()


def test_bad_expert_index_in_routing_is_reported(moe, ctx):
    T, k, E = 4, 2, 8
    topk = torch.tensor([[0, 1], [2, 3], [4, E + 3], [6, 7]], dtype=torch.int32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pairs = torch.empty(T * k, dtype=torch.int32, device="cuda")
    ws = moe.workspace(moe.bucket_tokens_ws_bytes(T, k, E))
    moe.moe_bucket_tokens(ctx, topk, E, counts, offsets, pairs, ws)
    with pytest.raises(moe.MoeError) as ei:
        ctx.check()
    assert ei.value.name == "MOE_ERR_BAD_EXPERT_INDEX" and ei.value.detail == E + 3


def test_host_validation(moe, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = si.get_workload("tiny")
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    out = torch.empty((r.T, r.d), device="cuda")
    need = moe.layer_forward_ws_bytes(layer, r.T)
    small = moe.workspace(need - 256)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(ctx, layer, x, out, small)
    assert ei.value.name == "MOE_ERR_WORKSPACE"
    ws = moe.workspace(need)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(ctx, layer, x, x, ws)  # out aliases x
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    topk = torch.empty((r.T, r.E + 1), dtype=torch.int32, device="cuda")
    gates = torch.empty((r.T, r.E + 1), device="cuda")
    wsr = moe.workspace(1 << 20)
    with pytest.raises(moe.MoeError) as ei:  # k > E
        moe.moe_route_topk(ctx, x, layer.router_w, None, r.E + 1, topk, gates, wsr)
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    xo = torch.empty((2, 100), device="cuda")
    with pytest.raises(moe.MoeError) as ei:  # d not a multiple of 32
        moe.moe_route_topk(ctx, xo, torch.empty((16, 100), device="cuda"), None, 4, topk, gates, wsr)
    assert ei.value.name == "MOE_ERR_UNSUPPORTED"
    # T = 0 is a no-op
    moe.moe_layer_forward(ctx, layer, x[:0], out[:0], ws)
    ctx.check()


def test_zero_gate_experts_with_nan_records_contribute_nothing(moe, ctx):
    # a +2000 bias on one expert: its gate is 1 and the other selected gates are
    # exactly 0, so their (NaN-scaled) records must not reach the output
    import oracle
    from quantized_expert_ffn_score_gb300 import synthetic
    from tests import gpu_util as gu
    r = si.get_workload("tiny")
    layer = synthetic.device_layer(r)
    bias = torch.zeros(r.E, device="cuda")
    bias[5] = 2000.0
    layer.struct.router_bias = bias.data_ptr()
    x = synthetic.device_x(r)
    topk = torch.empty((r.T, r.k), dtype=torch.int32, device="cuda")
    out = torch.empty((r.T, r.d), device="cuda")
    ws = moe.workspace(moe.layer_forward_ws_bytes(layer, r.T))
    moe.moe_layer_forward(ctx, layer, x, out, ws, topk_idx_out=topk)
    ctx.check()
    others = set(topk[:, 1:].cpu().numpy().reshape(-1).tolist()) - {5}
    gsz, ssz = r.ff * r.d // 2, r.ff * r.d // 32
    for e in others:  # poison the gate scales of every zero-gate expert
        layer.bank[e * layer.stride + gsz:e * layer.stride + gsz + ssz] = 255
    out2 = torch.empty_like(out)
    moe.moe_layer_forward(ctx, layer, x, out2, ws)
    ctx.check()
    assert torch.isfinite(out2).all()
    assert torch.equal(out, out2)
    xh = si.layer_x(r)
    recs = [si.layer_record(r, e) for e in range(r.E)]
    _, _, y, _ = oracle.layer_forward(xh, si.layer_router_w(r), bias.cpu().numpy(), r.d, r.ff, r.E, r.k, recs)
    gu.assert_rms_close(out2.cpu().numpy().astype(np.float64) - xh, y)


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable(moe):
    ctx = moe.Context(0)
    try:
        ctx.set_wait_limit_ns(2_000_000)  # 2 ms
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ctx.wait_selftest()  # a barrier nothing completes
        with pytest.raises(moe.MoeError) as ei:
            ctx.check()
        elapsed = time.perf_counter() - t0
        assert ei.value.name == "MOE_ERR_TIMEOUT" and ei.value.detail == -1
        assert elapsed < 1.0, f"the 2 ms limit was not applied ({elapsed:.3f} s)"
        ctx.check()  # the error word was cleared
        # the same context still runs the layer, with the short limit in force
        gu.full_check(moe, ctx, si.get_workload("tiny"))
        gu.full_check(moe, ctx, si.LayerRecipe("mid_wait_limit", d=1024, ff=576, E=40, k=6, T=37, seed=11,
                                               scale_lo=118, scale_hi=121))
        # 0 restores the default limit of 2 s
        ctx.set_wait_limit_ns(0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ctx.wait_selftest()
        with pytest.raises(moe.MoeError) as ei:
            ctx.check()
        elapsed = time.perf_counter() - t0
        assert ei.value.name == "MOE_ERR_TIMEOUT" and 1.9 <= elapsed < 10.0
        ctx.check()
    finally:
        ctx.close()
