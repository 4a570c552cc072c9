"""Helpers for the GPU parity tests: run a layer through the C ABI, run the
oracle on the same seeded inputs, compare.

Tolerance: max |y_gpu - y_ref| <= 2e-3 * RMS(y_ref) on the MoE delta y (the
layer output minus the residual), the bound the fp32-accumulating path must
meet; routing indices and bucket contents are compared bit for bit.
"""
import os

import numpy as np

import oracle
import seeded_inputs as si

TOL = 2e-3
NTHREADS = max(1, min(32, os.cpu_count() or 1))

# Achieved parity margins of this session: case name -> (max|err| / RMS,
# max|err|, RMS, tokens compared).  conftest.py writes them to the JSON file
# named by MOE_PARITY_MARGINS at the end of the session.
MARGINS = {}


def record_margin(name, err, rms, tokens):
    MARGINS[name] = {"max_err_over_rms": err / rms if rms > 0 else float("inf"), "max_abs_err": err, "rms": rms,
                     "tokens_compared": int(tokens)}


def rms_err(y_gpu, y_ref):
    rms = float(np.sqrt(np.mean(np.asarray(y_ref, dtype=np.float64) ** 2)))
    err = float(np.max(np.abs(np.asarray(y_gpu, dtype=np.float64) - y_ref)))
    return err, rms


def assert_rms_close(y_gpu, y_ref, tol=TOL, what="output"):
    err, rms = rms_err(y_gpu, y_ref)
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite values"
    assert err <= tol * rms, f"{what}: max|err| {err:.3e} > {tol} x RMS {rms:.3e} ({err / rms:.2e})"
    return err / rms


def x_host_f64(x):
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def oracle_layer(r, x_host, tokens=None, nthreads=NTHREADS, records=None):
    """(logits, topk, gates, y_delta, out) of the oracle; only `tokens` (default
    all) get expert outputs, and only their experts' records are generated."""
    W = si.layer_router_w(r)
    b = si.layer_bias(r)
    logits, idx, g = oracle.router(x_host, W, b, r.k, bias_mode=r.bias_mode)
    T = x_host.shape[0]
    mask = None
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    if tokens is not None:
        mask = np.zeros(T, dtype=np.uint8)
        mask[sel] = 1
    if records is None:
        needed = set(int(e) for e in idx[sel].reshape(-1)) | set(range(r.E, r.E + r.n_shared))
        records = si.layer_records(r, needed, nthreads=nthreads)
    cbs = None
    if r.quant == "rvq3":
        cb = si.layer_codebooks(r)
        cbs = (cb, cb, cb)
    idx2, g2, y, out = oracle.layer_forward(x_host, W, b, r.d, r.ff, r.E, r.k, records, quant=r.quant, act_kind=r.act,
                                            codebooks=cbs, token_mask=mask, nthreads=nthreads, n_shared=r.n_shared,
                                            bias_mode=r.bias_mode)
    assert np.array_equal(idx2, idx)
    return logits, idx, g, y, out


def gate_tolerance(r, x_host, logits_ref):
    """Bound on |g_gpu - g_ref| / g_ref from the fp32 logit error bound used by
    the router (gamma * ||W_e|| * ||x_t|| + 2^-23 |l|), applied to the logit
    differences inside the softmax, plus fp32 rounding of the gates.  With a
    bias, |l| is bounded by |key| + |bias| (logits_ref are the selection keys)."""
    W = x_host_f64(si.layer_router_w(r))
    xs = x_host_f64(x_host)
    nw = np.sqrt((W ** 2).sum(axis=1))
    nx = np.sqrt((xs ** 2).sum(axis=1))
    N = 8 if r.w_dtype == "bf16" else 4
    h = -(-r.d // (32 * N)) + (3 if N == 8 else 2) + 5 + (0 if (r.x_dtype == "bf16" and r.w_dtype == "bf16") else 1)
    u = 2.0 ** -24
    gamma = h * u / (1 - h * u) * 1.002 + 1e-12
    b = si.layer_bias(r)
    babs = 0.0 if b is None else np.abs(b.astype(np.float64))[None, :]
    beta = gamma * nx[:, None] * nw[None, :] + 1.2e-7 * (np.abs(logits_ref) + babs)
    return 2 * beta.max(axis=1) * 2 + 1e-6  # per token, relative


def check_routing(topk_gpu, gates_gpu, idx_ref, g_ref, rel_tol):
    np.testing.assert_array_equal(topk_gpu, idx_ref)
    rel = np.abs(gates_gpu.astype(np.float64) - g_ref) / g_ref
    assert np.all(rel <= np.asarray(rel_tol)[:, None]), f"gate error {rel.max():.3e}"


def run_layer(moe, ctx, layer, x, out_dtype=None):
    import torch
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    T = x.shape[0]
    r = layer.recipe
    ks = r.k + r.n_shared  # the routed slots, then the shared experts
    out = torch.empty((T, r.d), dtype=out_dtype, device="cuda")
    topk = torch.full((T, ks), -1, dtype=torch.int32, device="cuda")
    gates = torch.empty((T, ks), dtype=torch.float32, device="cuda")
    counts = torch.empty(r.E + r.n_shared, dtype=torch.int32, device="cuda")
    ws = moe.workspace(moe.layer_forward_ws_bytes(layer, T))
    moe.moe_layer_forward(ctx, layer, x, out, ws, topk_idx_out=topk, gates_out=gates, counts_out=counts)
    ctx.check()
    return out.float().cpu().numpy(), topk.cpu().numpy(), gates.cpu().numpy(), counts.cpu().numpy()


def full_check(moe, ctx, r, tokens=None):
    from quantized_expert_ffn_score_gb300 import synthetic
    layer = synthetic.device_layer(r)
    x = synthetic.device_x(r)
    out, topk, gates, counts = run_layer(moe, ctx, layer, x)
    xh = si.layer_x(r)
    logits, idx, g, y, o = oracle_layer(r, xh, tokens=tokens)
    check_routing(topk[:, :r.k], gates[:, :r.k], idx, g, gate_tolerance(r, xh, logits))
    # shared experts close every row with gate 1
    np.testing.assert_array_equal(topk[:, r.k:], np.broadcast_to(np.arange(r.E, r.E + r.n_shared), (r.T, r.n_shared)))
    assert np.all(gates[:, r.k:] == 1.0)
    np.testing.assert_array_equal(counts, np.bincount(topk.reshape(-1), minlength=r.E + r.n_shared))
    np.testing.assert_array_equal(counts[:r.E], np.bincount(idx.reshape(-1), minlength=r.E))
    sel = np.arange(r.T) if tokens is None else np.asarray(tokens)
    delta = out[sel].astype(np.float64) - x_host_f64(xh)[sel]
    err, rms = rms_err(delta, y[sel])
    record_margin(r.name, err, rms, len(sel))
    rel = assert_rms_close(delta, y[sel], what=r.name)
    return rel, counts
