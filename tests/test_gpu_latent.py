"""The latent projections either side of the routed experts (moe_project,
moe_latent_layer_forward) against the fp64 oracle, through the C ABI.  The
pages give the latent width (3584) but not K3's hidden width, so the tests
run the latent layer at two stated hidden widths, 1536 and 2048, around a
1024-wide latent layer (and 4096 at one token).

moe_project: every output within the fp32 summation bound of the oracle's
fp64 sum (K u sum_k |W[n][k] x[t][k]|), for bf16 and fp32 operands, ragged
row counts and K.  The latent layer: the latent input z = bf16(W_in x) may
differ from the oracle's rounding of its fp64 projection only by one bf16
step where the two sums straddle a rounding boundary; the rest of the layer
is compared teacher-forced on the GPU's z (routing bit-exact, the MoE part
of the output within 2e-3 x RMS)."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

LATENT = si.LayerRecipe("latent_mid", d=1024, ff=576, E=40, k=6, T=37, seed=91, scale_lo=118, scale_hi=121)


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


_TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


def _dev(a, dt):
    a = np.ascontiguousarray(a)
    if dt == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


@pytest.mark.parametrize("T,K,N,xdt,wdt", [(1, 1024, 99, "bf16", "bf16"), (5, 1056, 128, "f32", "bf16"),
                                           (37, 512, 61, "bf16", "f32"), (9, 2048, 40, "f32", "f32")])
def test_project_matches_oracle(lib, ctx, T, K, N, xdt, wdt):
    x = si.normal(51, 1, 1.0, T * K, xdt).reshape(T, K)
    W = si.normal(51, 2, 1.0 / np.sqrt(K), N * K, wdt).reshape(N, K)
    resid = si.normal(51, 3, 1.0, T * N, "f32").reshape(T, N)
    y = torch.empty((T, N), dtype=torch.float32, device="cuda")
    lib.moe_project(ctx, _dev(x, xdt), _dev(W, wdt), y, resid=_dev(resid, "f32"))
    ctx.check()
    ref = oracle.project(x, W) + resid
    xf = gu.x_host_f64(x)
    wf = gu.x_host_f64(W)
    bound = K * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T) + 2.0 ** -24 * np.abs(resid) + 1e-30
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"max err / bound {np.max(err / bound):.3f}"
    # bf16 output: the fp32 result rounded to nearest even
    yb = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    lib.moe_project(ctx, _dev(x, xdt), _dev(W, wdt), yb, resid=_dev(resid, "f32"))
    ctx.check()
    np.testing.assert_array_equal(yb.view(torch.int16).cpu().numpy(), y.to(torch.bfloat16).view(torch.int16).cpu().numpy())


def _latent_weights(r, D, seed):
    w_in = si.normal(seed, 91, 1.0 / np.sqrt(D), r.d * D, "bf16").reshape(r.d, D)
    w_out = si.normal(seed, 92, 1.0 / np.sqrt(r.d), D * r.d, "bf16").reshape(D, r.d)
    x = si.normal(seed, 90, 1.0, r.T * D, "bf16").reshape(r.T, D)
    return x, w_in, w_out


@pytest.mark.parametrize("D,T", [(1536, 37), (2048, 37), (4096, 1)])
def test_latent_layer_matches_oracle(lib, ctx, D, T):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = LATENT.with_(T=T, name=f"latent_mid_D{D}_T{T}")
    layer = synthetic.device_layer(r)
    x, w_in, w_out = _latent_weights(r, D, seed=93 + D)
    out = torch.empty((T, D), dtype=torch.float32, device="cuda")
    z = torch.empty((T, r.d), dtype=torch.bfloat16, device="cuda")
    ws = lib.workspace(lib.latent_layer_forward_ws_bytes(layer, D, T))
    lib.moe_latent_layer_forward(ctx, layer, _dev(w_in, "bf16"), _dev(w_out, "bf16"), _dev(x, "bf16"), out, ws,
                                 latent_out=z)
    ctx.check()
    zb = z.view(torch.int16).cpu().numpy().view(np.uint16)
    # 1. the latent input against the oracle's rounding of its fp64 projection
    zr = oracle.project(x, w_in)
    z_or = oracle.round_bf16(zr)
    diff = zb != z_or
    if np.any(diff):  # only one bf16 step apart, and only where the fp32 sum's error bound reaches the boundary
        zg = gu.x_host_f64(zb[diff])
        zo = gu.x_host_f64(z_or[diff])
        step = np.maximum(np.abs(zo), np.abs(zg)) * 2.0 ** -7
        assert np.all(np.abs(zg - zo) <= step * 1.001)
        absdot = (np.abs(gu.x_host_f64(x)) @ np.abs(gu.x_host_f64(w_in)).T)[diff]
        assert np.all(np.abs(zr[diff] - (zg + zo) / 2) <= D * 2.0 ** -24 * absdot + 1e-30)
    assert diff.mean() < 0.01
    # 2. routing of the GPU's z: bit-exact against the oracle's
    topk = torch.empty((T, r.k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, r.k), dtype=torch.float32, device="cuda")
    lib.moe_route_topk(ctx, z, layer.router_w, None, r.k, topk, gates,
                       lib.workspace(lib.route_topk_ws_bytes(T, r.d, r.E, r.k)))
    ctx.check()
    logits, idx, g, y, _ = gu.oracle_layer(r, zb)
    gu.check_routing(topk.cpu().numpy(), gates.cpu().numpy(), idx, g, gu.gate_tolerance(r, zb, logits))
    # 3. the output: x + W_out (MoE delta of the GPU's z)
    moe_part = out.cpu().numpy().astype(np.float64) - gu.x_host_f64(x)
    ref = y @ gu.x_host_f64(w_out).T
    err, rms = gu.rms_err(moe_part, ref)
    gu.record_margin(r.name, err, rms, T)
    gu.assert_rms_close(moe_part, ref, what=r.name)


def test_latent_layer_validation(lib, ctx):
    from quantized_expert_ffn_score_gb300 import synthetic
    r = LATENT.with_(T=2)
    layer = synthetic.device_layer(r)
    D = 1536
    x = torch.zeros((2, D), dtype=torch.bfloat16, device="cuda")
    w_in = torch.zeros((r.d, D), dtype=torch.bfloat16, device="cuda")
    w_out = torch.zeros((D, r.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((2, D), dtype=torch.float32, device="cuda")
    assert lib.latent_layer_forward_ws_bytes(layer, 100, 2) == 0  # D not a multiple of 32
    ws = lib.workspace(lib.latent_layer_forward_ws_bytes(layer, D, 2))
    with pytest.raises(lib.MoeError) as ei:
        lib.moe_latent_layer_forward(ctx, layer, w_in, w_out, x, out, ws[:1024])
    assert ei.value.name == "MOE_ERR_WORKSPACE"
    with pytest.raises(lib.MoeError):
        lib.moe_project(ctx, x[:, :1000], w_in[:, :1000], out)  # K not a multiple of 32
