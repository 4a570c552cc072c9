"""The six-layer K3 stack (896 MXFP4 experts per layer, ~94 GB resident, 64
tokens): every layer on its own seeded input against the oracle, then the
chained stack against the oracle's own chain.

In the chain each layer's input is the previous layer's output rounded to
bf16.  The GPU's fp32 output and the oracle's fp64 output round to different
bf16 values for a few elements (those within an fp32 error of a rounding
boundary), so later layers see inputs that differ by one bf16 unit in a few
places and a near-tie in the router may flip.  Such a flip is accepted only if
the oracle's own logit gap between the swapped experts is within the change
the input difference can cause (Cauchy-Schwarz: |dl_e| <= ||W_e|| ||dx||);
that token is then no longer compared.  Layer 0 (identical inputs) is held to
the parity tolerance; later layers' deviations are reported (and guarded
against gross errors only), since the two chains' inputs legitimately differ.
Each layer's own parity at full size, on all 64 tokens, is the first test; the
stack call's routing trace must equal the layer-by-layer routing."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from seeded_inputs.workloads import STACK_LAYERS, STACK_T, stack_layer
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLE = [0, 37]


@pytest.fixture(scope="module")
def moe():
    from quantized_expert_ffn_score_gb300 import build, moe
    build.build()
    return moe


def _gpu_layer(moe, ctx, layer, x, out_dtype):
    r = layer.recipe
    T = x.shape[0]
    out = torch.empty((T, r.d), dtype=out_dtype, device="cuda")
    topk = torch.empty((T, r.k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, r.k), dtype=torch.float32, device="cuda")
    moe.moe_layer_forward(ctx, layer, x, out, moe.workspace(moe.layer_forward_ws_bytes(layer, T)), topk_idx_out=topk,
                          gates_out=gates)
    ctx.check()
    return out, topk.cpu().numpy(), gates.cpu().numpy()


def _bf16_bits(a32):
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_each_stack_layer_on_its_own_input(moe):
    # every one of the 64 tokens of every layer: routing bit-exact, outputs
    # within 2e-3 x RMS of the oracle's
    from quantized_expert_ffn_score_gb300 import synthetic
    ctx = moe.Context(0)
    for l in range(STACK_LAYERS):
        r = stack_layer(l)
        layer = synthetic.device_layer(r)
        x = synthetic.device_x(r)
        out, topk, gates = _gpu_layer(moe, ctx, layer, x, torch.float32)
        xh = si.layer_x(r)
        logits, idx, g, y, _ = gu.oracle_layer(r, xh)
        gu.check_routing(topk, gates, idx, g, gu.gate_tolerance(r, xh, logits))
        delta = out.cpu().numpy().astype(np.float64) - gu.x_host_f64(xh)
        err, rms = gu.rms_err(delta, y)
        gu.record_margin(r.name, err, rms, r.T)
        gu.assert_rms_close(delta, y, what=f"stack layer {l}")
        del layer
        torch.cuda.empty_cache()
    ctx.close()


def test_chained_stack_against_the_oracle_chain(moe):
    from quantized_expert_ffn_score_gb300 import synthetic
    ctx = moe.Context(0)
    recipes = [stack_layer(l) for l in range(STACK_LAYERS)]
    layers = [synthetic.device_layer(r) for r in recipes]
    x0 = synthetic.device_x(recipes[0])
    # the library's stack call (with its routing trace) and the same chain
    # layer by layer agree bit for bit
    out_stack = torch.empty((STACK_T, recipes[0].d), dtype=torch.float32, device="cuda")
    k = recipes[0].k
    trace = torch.full((STACK_LAYERS, STACK_T, k), -1, dtype=torch.int32, device="cuda")
    moe.moe_stack_forward_ex(ctx, layers, x0, out_stack, moe.workspace(moe.stack_forward_ws_bytes(layers, STACK_T)),
                             topk_trace=trace)
    ctx.check()
    trace = trace.cpu().numpy()
    x = x0
    gpu_in, gpu_topk, gpu_out = [], [], []
    for l, layer in enumerate(layers):
        last = l == STACK_LAYERS - 1
        gpu_in.append(x.view(torch.int16).cpu().numpy().view(np.uint16)[SAMPLE])
        out, topk, _ = _gpu_layer(moe, ctx, layer, x, torch.float32)
        np.testing.assert_array_equal(trace[l], topk)
        gpu_topk.append(topk[SAMPLE])
        gpu_out.append(out.cpu().numpy()[SAMPLE])
        x = out if last else out.to(torch.bfloat16)
    assert torch.equal(x, out_stack)
    # the oracle's own chain on the sampled tokens
    x_or = si.layer_x(recipes[0])[SAMPLE]
    alive = np.ones(len(SAMPLE), dtype=bool)
    flips = 0
    dev = []  # (layer, token, max|err| / RMS) of the free-running comparison
    for l, r in enumerate(recipes):
        W = si.layer_router_w(r)
        logits, idx, g = oracle.router(x_or, W, None, r.k)
        for s in range(len(SAMPLE)):
            if alive[s] and not np.array_equal(idx[s], gpu_topk[l][s]):
                # accept only a near-tie the input difference explains
                dx = gu.x_host_f64(gpu_in[l][s]) - gu.x_host_f64(x_or[s])
                wn = np.sqrt((gu.x_host_f64(W) ** 2).sum(axis=1))
                swapped = set(idx[s].tolist()) ^ set(gpu_topk[l][s].tolist())
                moved = [e for e in range(r.k) if idx[s][e] != gpu_topk[l][s][e]]
                cand = sorted(swapped | {int(idx[s][e]) for e in moved} | {int(gpu_topk[l][s][e]) for e in moved})
                lv = logits[s][cand]
                gap = lv.max() - lv.min()
                allow = 2 * wn[cand].max() * np.linalg.norm(dx) + 1e-6
                assert gap <= allow, f"layer {l} token {SAMPLE[s]}: routing differs beyond a near-tie"
                alive[s] = False
                flips += 1
        recs = {}
        for s in np.nonzero(alive)[0]:
            for e in idx[s]:
                recs.setdefault(int(e), None)
        records = [si.layer_record(r, e) if e in recs else None for e in range(r.E)]
        mask = alive.astype(np.uint8)
        _, _, y, out_or = oracle.layer_forward(x_or, W, None, r.d, r.ff, r.E, r.k, records, token_mask=mask,
                                               nthreads=gu.NTHREADS)
        for s in np.nonzero(alive)[0]:
            y_gpu = gpu_out[l][s].astype(np.float64) - gu.x_host_f64(gpu_in[l][s])
            if l == 0:  # identical inputs: the parity tolerance
                gu.assert_rms_close(y_gpu, y[s], what=f"chained layer 0 token {SAMPLE[s]}")
            else:  # inputs differ by bf16 rounding: reported, guarded only against gross errors
                err, rms = gu.rms_err(y_gpu, y[s])
                dev.append((l, SAMPLE[s], err / rms))
                assert err <= 5e-2 * rms, f"chained layer {l} token {SAMPLE[s]}: deviation {err / rms:.2e} x RMS"
        # next layer's input: the fp64 output rounded to fp32, then to bf16 (nearest even)
        nxt = x_or.copy()
        for s in np.nonzero(alive)[0]:
            nxt[s] = _bf16_bits(out_or[s].astype(np.float32))
        x_or = nxt
    print(f"free-running stack: {flips} routing flip(s) among {len(SAMPLE)} sampled tokens; "
          f"deviation per (layer, token): {[(l, t, round(v, 5)) for l, t, v in dev]}")
    ctx.close()
