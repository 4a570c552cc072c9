"""moe_stack_forward_ex: a stack of layers with the routing every layer took
(top-k experts, gates and tokens per expert), through the C ABI.

The trace must equal, bit for bit, what moe_layer_forward returns for the same
layer on the same input (the stack feeds each layer the bf16 rounding of the
previous layer's output), and every layer's traced routing must equal the
oracle's routing of that layer's input (teacher-forced: the oracle is given
the GPU's bf16 layer input), for every token.  The output must be the one of
moe_stack_forward."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

BASE = si.LayerRecipe("stack_trace", d=1024, ff=576, E=40, k=6, T=29, seed=70, scale_lo=118, scale_hi=121)


@pytest.fixture(scope="module")
def lib():
    from quantized_expert_ffn_score_gb300 import build, moe
    build.build()
    return moe


def _recipes():
    # three layers: plain; 2 shared experts with the selection-only bias; SiTU
    return [BASE.with_(seed=70), BASE.with_(seed=71, n_shared=2, bias="zipf", bias_mode="select"),
            BASE.with_(seed=72, act="situ")]


def test_trace_matches_layer_calls_and_oracle_routing(lib):
    from quantized_expert_ffn_score_gb300 import synthetic
    ctx = lib.Context(0)
    recipes = _recipes()
    layers = [synthetic.device_layer(r) for r in recipes]
    T, d = BASE.T, BASE.d
    x0 = synthetic.device_x(recipes[0])
    ks = [r.k + r.n_shared for r in recipes]
    Es = [r.E + r.n_shared for r in recipes]
    topk_tr = torch.full((T * sum(ks),), -1, dtype=torch.int32, device="cuda")
    gates_tr = torch.full((T * sum(ks),), float("nan"), dtype=torch.float32, device="cuda")
    counts_tr = torch.full((sum(Es),), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((T, d), dtype=torch.float32, device="cuda")
    ws = lib.workspace(lib.stack_forward_ws_bytes(layers, T))
    lib.moe_stack_forward_ex(ctx, layers, x0, out, ws, topk_trace=topk_tr, gates_trace=gates_tr,
                             counts_trace=counts_tr)
    ctx.check()
    out_plain = torch.empty_like(out)
    lib.moe_stack_forward(ctx, layers, x0, out_plain, ws)
    ctx.check()
    assert torch.equal(out, out_plain)
    # layer by layer, each fed the bf16 rounding of the previous output
    x = x0
    po, eo = 0, 0
    for l, (r, layer) in enumerate(zip(recipes, layers)):
        o, topk, gates, counts = gu.run_layer(lib, ctx, layer, x)
        n = T * ks[l]
        np.testing.assert_array_equal(topk_tr[po:po + n].cpu().numpy().reshape(T, ks[l]), topk)
        np.testing.assert_array_equal(gates_tr[po:po + n].cpu().numpy().reshape(T, ks[l]), gates)
        np.testing.assert_array_equal(counts_tr[eo:eo + Es[l]].cpu().numpy(), counts)
        # the oracle's routing of this layer's input (teacher-forced), every token
        xh = x.cpu().numpy() if x.dtype == torch.float32 else x.view(torch.int16).cpu().numpy().view(np.uint16)
        logits, idx, g = oracle.router(xh, si.layer_router_w(r), si.layer_bias(r), r.k, bias_mode=r.bias_mode)
        gu.check_routing(topk[:, :r.k], gates[:, :r.k], idx, g, gu.gate_tolerance(r, xh, logits))
        po += n
        eo += Es[l]
        x = torch.from_numpy(o).cuda().to(torch.bfloat16) if l < len(recipes) - 1 else None
    ctx.close()
