"""Device-resident synthetic layers built from the seeded workload recipes.

Everything is generated in HBM by the seeded-input generator's device filler,
so the host never holds the expert banks (15.7 GB per K3 layer).  Records are
placed at a 4 KiB stride in one allocation, and the record pointer table lives
on the device.
"""
import numpy as np
import torch

import seeded_inputs as si

from . import moe

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def record_stride(r):
    b = si.record_size(r)
    return (b + 4095) // 4096 * 4096


def device_layer(r, device="cuda", missing=()):
    """Builds layer recipe `r` on the device (E routed records, then the
    n_shared shared ones); experts listed in `missing` get a NULL record
    pointer."""
    stream = torch.cuda.current_stream().cuda_stream
    W = torch.empty((r.E, r.d), dtype=_DT[r.w_dtype], device=device)
    si.dev_layer_router_w(r, W.data_ptr(), cuda_stream=stream)
    bias = None
    b = si.layer_bias(r)
    if b is not None:
        bias = torch.from_numpy(b).to(device)
    stride = record_stride(r)
    n_rec = r.E + r.n_shared
    bank = torch.empty(stride * n_rec, dtype=torch.uint8, device=device)
    si.dev_record_bank(r, bank.data_ptr(), stride, n_exp=n_rec, cuda_stream=stream)
    ptrs = np.array([bank.data_ptr() + e * stride for e in range(n_rec)], dtype=np.int64)
    for e in missing:
        ptrs[e] = 0
    records = torch.from_numpy(ptrs).to(device)
    cbs = None
    keep = [bank]
    if r.quant == "rvq3":
        cb = torch.empty(3 * 256 * 8, dtype=torch.int16, device=device)
        si.dev_layer_codebooks(r, cb.data_ptr(), cuda_stream=stream)
        cbs = (cb, cb, cb)
    layer = moe.Layer(r.d, r.ff, r.E, r.k, W, records, quant=r.quant, act=r.act, router_bias=bias, codebooks=cbs,
                      keep=keep, n_shared=r.n_shared, bias_mode=r.bias_mode)
    layer.bank = bank
    layer.stride = stride
    layer.recipe = r
    return layer


def device_x(r, T=None, token_offset=0, device="cuda"):
    T = r.T if T is None else T
    x = torch.empty((T, r.d), dtype=_DT[r.x_dtype], device=device)
    si.dev_layer_x(r, x.data_ptr(), T=T, token_offset=token_offset, cuda_stream=torch.cuda.current_stream().cuda_stream)
    return x


def host_x(r, T=None, token_offset=0):
    """The same x on the host (numpy: float32 or bf16 bit patterns in uint16)."""
    return si.layer_x(r, T=T, token_offset=token_offset)
