"""Thin ctypes binding of libmoe_gb300.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory and
streams); integer arguments are passed through.  If the library has not been
built this module raises on first use -- there is no fallback path.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_BAD_EXPERT_INDEX", 6: "MOE_ERR_MISSING_EXPERT", 7: "MOE_ERR_TIMEOUT",
          8: "MOE_ERR_BAD_RECORD"}
MOE_F32, MOE_BF16 = 0, 1
ACT = {"swiglu": 0, "situ": 1}
QUANT = {"mxfp4": 0, "rvq3": 1}
BIAS_MODE = {"logit": 0, "select": 1}
MXFP4_KERNEL = {"block_scaled": 0, "gemv": 1, "auto": 2}

# every symbol include/moe.h declares
EXPORTS = ["moe_status_str", "moe_version", "moe_ctx_create", "moe_ctx_destroy", "moe_ctx_check", "moe_ctx_num_sms",
           "moe_ctx_set_mxfp4_kernel", "moe_ctx_mxfp4_kernel",
           "moe_ctx_profile", "moe_ctx_profile_read", "moe_ctx_stats",
           "moe_mxfp4_record_bytes", "moe_rvq3_record_bytes", "moe_route_topk_ws_bytes", "moe_bucket_tokens_ws_bytes",
           "moe_expert_ffn_ws_bytes", "moe_layer_forward_ws_bytes", "moe_stack_forward_ws_bytes", "moe_route_topk",
           "moe_route_topk_ex",
           "moe_bucket_tokens", "moe_expert_ffn_mxfp4", "moe_expert_ffn_rvq3", "moe_combine", "moe_layer_forward",
           "moe_stack_forward", "moe_stack_forward_ex", "moe_expert_ffn_mxfp4_static",
           "moe_expert_ffn_mxfp4_static_max_bytes", "moe_records_check_ws_bytes", "moe_records_check",
           "moe_ctx_set_wait_limit_ns", "moe_ctx_wait_selftest", "moe_rvq3_repack", "moe_tier_create",
           "moe_tier_destroy", "moe_tier_observe", "moe_tier_rebalance", "moe_tier_pin", "moe_tier_residency",
           "moe_tier_plan", "moe_project", "moe_latent_layer_forward_ws_bytes", "moe_latent_layer_forward"]


class MoeError(RuntimeError):
    def __init__(self, status, what, detail=None):
        self.status = status
        self.name = STATUS.get(status, str(status))
        self.detail = detail
        super().__init__(f"{what}: {self.name}" + (f" (detail {detail})" if detail is not None else ""))


class MxExperts(ctypes.Structure):
    _fields_ = [("records", ctypes.c_void_p), ("d", ctypes.c_int), ("ff", ctypes.c_int), ("E", ctypes.c_int)]


class RvqExperts(ctypes.Structure):
    _fields_ = [("records", ctypes.c_void_p), ("codebooks", ctypes.c_void_p * 3), ("d", ctypes.c_int),
                ("ff", ctypes.c_int), ("E", ctypes.c_int)]


class TierDesc(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("record_bytes", ctypes.c_size_t), ("host_records", ctypes.c_void_p),
                ("slots", ctypes.c_void_p), ("n_slots", ctypes.c_int), ("slot_stride", ctypes.c_size_t),
                ("records", ctypes.c_void_p), ("direct_host", ctypes.c_int), ("decay", ctypes.c_float)]


class LayerStruct(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("ff", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("act", ctypes.c_int), ("quant", ctypes.c_int), ("router_w", ctypes.c_void_p),
                ("router_w_dtype", ctypes.c_int), ("router_bias", ctypes.c_void_p), ("mxfp4", MxExperts),
                ("rvq3", RvqExperts), ("n_shared", ctypes.c_int), ("bias_mode", ctypes.c_int)]


_lib = None


def lib():
    """Loads the in-tree CUDA library; raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with quantized_expert_ffn_score_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_status_str.argtypes, L.moe_status_str.restype = [i32], ctypes.c_char_p
        L.moe_version.restype = ctypes.c_char_p
        L.moe_ctx_create.argtypes = [ctypes.POINTER(vp), i32]
        L.moe_ctx_destroy.argtypes = [vp]
        L.moe_ctx_destroy.restype = None
        L.moe_ctx_check.argtypes = [vp, vp, ctypes.POINTER(i32)]
        L.moe_ctx_num_sms.argtypes = [vp]
        L.moe_ctx_profile.argtypes, L.moe_ctx_profile.restype = [vp, i32], i32
        L.moe_ctx_stats.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong)]
        L.moe_ctx_stats.restype = i32
        L.moe_ctx_profile_read.argtypes = [vp, vp, i32, ctypes.c_char_p, ctypes.POINTER(i32),
                                           ctypes.POINTER(ctypes.c_double)]
        L.moe_ctx_profile_read.restype = i32
        L.moe_mxfp4_record_bytes.argtypes, L.moe_mxfp4_record_bytes.restype = [i32, i32], sz
        L.moe_rvq3_record_bytes.argtypes, L.moe_rvq3_record_bytes.restype = [i32, i32], sz
        L.moe_route_topk_ws_bytes.argtypes, L.moe_route_topk_ws_bytes.restype = [i32, i32, i32, i32], sz
        L.moe_bucket_tokens_ws_bytes.argtypes, L.moe_bucket_tokens_ws_bytes.restype = [i32, i32, i32], sz
        L.moe_expert_ffn_ws_bytes.argtypes, L.moe_expert_ffn_ws_bytes.restype = [i32, i32, i32, i32, i32, i32], sz
        L.moe_layer_forward_ws_bytes.argtypes = [ctypes.POINTER(LayerStruct), i32]
        L.moe_layer_forward_ws_bytes.restype = sz
        L.moe_stack_forward_ws_bytes.argtypes = [ctypes.POINTER(LayerStruct), i32, i32]
        L.moe_stack_forward_ws_bytes.restype = sz
        L.moe_route_topk.argtypes = [vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, sz, vp]
        L.moe_route_topk_ex.argtypes = [vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, vp, vp, vp, sz, vp]
        L.moe_bucket_tokens.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
        L.moe_expert_ffn_mxfp4.argtypes = [vp, vp, i32, i32, i32, ctypes.POINTER(MxExperts), i32, vp, vp, vp, vp, sz,
                                           vp]
        L.moe_expert_ffn_rvq3.argtypes = [vp, vp, i32, i32, i32, ctypes.POINTER(RvqExperts), i32, vp, vp, vp, vp, sz,
                                          vp]
        L.moe_combine.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, vp, i32, vp]
        L.moe_expert_ffn_mxfp4_static.argtypes = [vp, vp, i32, i32, i32, ctypes.POINTER(MxExperts), i32, vp, vp, vp,
                                                  vp]
        L.moe_expert_ffn_mxfp4_static.restype = i32
        L.moe_expert_ffn_mxfp4_static_max_bytes.restype = sz
        L.moe_records_check_ws_bytes.argtypes, L.moe_records_check_ws_bytes.restype = [i32, sz], sz
        L.moe_records_check.argtypes, L.moe_records_check.restype = [vp, vp, i32, sz, vp, vp, vp, sz, vp], i32
        L.moe_layer_forward.argtypes = [vp, ctypes.POINTER(LayerStruct), vp, i32, i32, vp, i32, vp, vp, vp, vp, sz,
                                        vp]
        L.moe_stack_forward.argtypes = [vp, ctypes.POINTER(LayerStruct), i32, vp, i32, i32, vp, i32, vp, sz, vp]
        L.moe_stack_forward_ex.argtypes = [vp, ctypes.POINTER(LayerStruct), i32, vp, i32, i32, vp, i32, vp, vp, vp, vp,
                                           sz, vp]
        L.moe_ctx_set_wait_limit_ns.argtypes = [vp, ctypes.c_ulonglong]
        L.moe_ctx_wait_selftest.argtypes = [vp, vp]
        L.moe_rvq3_repack.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.moe_tier_create.argtypes = [vp, ctypes.POINTER(TierDesc), ctypes.POINTER(vp)]
        L.moe_tier_destroy.argtypes, L.moe_tier_destroy.restype = [vp], None
        L.moe_tier_observe.argtypes = [vp, vp, vp]
        L.moe_tier_rebalance.argtypes = [vp, vp, ctypes.POINTER(i32)]
        L.moe_tier_pin.argtypes = [vp, vp, i32, vp]
        L.moe_tier_residency.argtypes = [vp, vp, vp]
        L.moe_tier_plan.argtypes, L.moe_tier_plan.restype = [i32, i32, vp, vp, vp, vp], i32
        L.moe_project.argtypes = [vp, vp, i32, i32, i32, vp, i32, i32, vp, i32, vp, i32, vp]
        L.moe_latent_layer_forward_ws_bytes.argtypes = [ctypes.POINTER(LayerStruct), i32, i32]
        L.moe_latent_layer_forward_ws_bytes.restype = sz
        L.moe_latent_layer_forward.argtypes = [vp, ctypes.POINTER(LayerStruct), vp, vp, i32, i32, vp, i32, i32, vp,
                                               i32, vp, vp, sz, vp]
        for f in ("moe_ctx_create", "moe_ctx_check", "moe_route_topk", "moe_route_topk_ex", "moe_bucket_tokens",
                  "moe_expert_ffn_mxfp4",
                  "moe_expert_ffn_rvq3", "moe_combine", "moe_layer_forward", "moe_stack_forward", "moe_stack_forward_ex",
                  "moe_ctx_set_wait_limit_ns", "moe_ctx_wait_selftest", "moe_rvq3_repack", "moe_tier_create",
                  "moe_tier_observe", "moe_tier_rebalance", "moe_tier_pin", "moe_tier_residency", "moe_project",
                  "moe_latent_layer_forward"):
            getattr(L, f).restype = i32
        L.moe_ctx_num_sms.restype = i32
        L.moe_ctx_set_mxfp4_kernel.argtypes, L.moe_ctx_set_mxfp4_kernel.restype = [vp, i32], i32
        L.moe_ctx_mxfp4_kernel.argtypes, L.moe_ctx_mxfp4_kernel.restype = [vp], i32
        _lib = L
    return _lib


def version():
    return lib().moe_version().decode()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dt(t):
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    raise TypeError(f"unsupported activation dtype {t.dtype}")


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream if hasattr(s, "cuda_stream") else s


def _check(rc, what):
    if rc != MOE_OK:
        raise MoeError(rc, what)


class Context:
    """Owns a moe_ctx (its device error word)."""

    def __init__(self, device=None):
        dev = torch.cuda.current_device() if device is None else device
        h = ctypes.c_void_p()
        _check(lib().moe_ctx_create(ctypes.byref(h), dev), "moe_ctx_create")
        self.handle = h
        self.device = dev

    @property
    def num_sms(self):
        return lib().moe_ctx_num_sms(self.handle)

    def check(self, stream=None):
        """Synchronises the stream; raises MoeError if a kernel flagged an error."""
        detail = ctypes.c_int(-1)
        rc = lib().moe_ctx_check(self.handle, _stream(stream), ctypes.byref(detail))
        if rc != MOE_OK:
            raise MoeError(rc, "device error", detail.value)

    def stats(self, stream=None):
        """(tokens that needed the fp64 top-k recheck, logits recomputed sequentially) since the last call."""
        a, b = ctypes.c_longlong(0), ctypes.c_longlong(0)
        _check(lib().moe_ctx_stats(self.handle, _stream(stream), ctypes.byref(a), ctypes.byref(b)), "moe_ctx_stats")
        return a.value, b.value

    @property
    def mxfp4_kernel(self):
        """'auto' (default), 'block_scaled' (tensor-core MMA on the stored codes and scales) or 'gemv'."""
        v = lib().moe_ctx_mxfp4_kernel(self.handle)
        return {k: n for n, k in MXFP4_KERNEL.items()}.get(v, v)

    @mxfp4_kernel.setter
    def mxfp4_kernel(self, name):
        _check(lib().moe_ctx_set_mxfp4_kernel(self.handle, MXFP4_KERNEL[name]), "moe_ctx_set_mxfp4_kernel")

    def set_wait_limit_ns(self, ns):
        """Limit of the kernels' pipeline waits in ns (0: the default, 2 s)."""
        _check(lib().moe_ctx_set_wait_limit_ns(self.handle, int(ns)), "moe_ctx_set_wait_limit_ns")

    def wait_selftest(self, stream=None):
        """Launches a wait that nothing completes; it times out after the wait
        limit and the next check() raises MOE_ERR_TIMEOUT."""
        _check(lib().moe_ctx_wait_selftest(self.handle, _stream(stream)), "moe_ctx_wait_selftest")

    def profile(self, capacity):
        """Turns per-launch event timing on (capacity launches between reads) or off (0)."""
        _check(lib().moe_ctx_profile(self.handle, capacity), "moe_ctx_profile")

    def profile_read(self, stream=None, max_entries=32):
        """{kernel name: (launches, total ms)} since the last read."""
        names = ctypes.create_string_buffer(32 * max_entries)
        launches = (ctypes.c_int * max_entries)()
        ms = (ctypes.c_double * max_entries)()
        n = lib().moe_ctx_profile_read(self.handle, _stream(stream), max_entries, names, launches, ms)
        if n < 0:
            raise MoeError(-n, "moe_ctx_profile_read")
        raw = names.raw
        return {raw[32 * i:32 * i + 32].split(b"\0")[0].decode(): (launches[i], ms[i]) for i in range(n)}

    def close(self):
        if self.handle:
            lib().moe_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------------------------------- sizes

def mxfp4_record_bytes(d, ff):
    return int(lib().moe_mxfp4_record_bytes(d, ff))


def rvq3_record_bytes(d, ff):
    return int(lib().moe_rvq3_record_bytes(d, ff))


def route_topk_ws_bytes(T, d, E, k):
    return int(lib().moe_route_topk_ws_bytes(T, d, E, k))


def bucket_tokens_ws_bytes(T, k, E):
    return int(lib().moe_bucket_tokens_ws_bytes(T, k, E))


def expert_ffn_ws_bytes(T, k, d, ff, E, quant="mxfp4"):
    return int(lib().moe_expert_ffn_ws_bytes(T, k, d, ff, E, QUANT[quant]))


def layer_forward_ws_bytes(layer, T):
    return int(lib().moe_layer_forward_ws_bytes(ctypes.byref(layer.struct), T))


def stack_forward_ws_bytes(layers, T):
    arr = (LayerStruct * len(layers))(*[l.struct for l in layers])
    return int(lib().moe_stack_forward_ws_bytes(arr, len(layers), T))


def workspace(nbytes, device=None):
    """A 256-byte aligned uint8 CUDA buffer (torch allocations are 512-byte aligned)."""
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device or "cuda")


# ----------------------------------------------------------------------------- experts / layer

class Layer:
    """A moe_layer: keeps the tensors it points at alive.  records: device
    array of E + n_shared record pointers (the shared experts last)."""

    def __init__(self, d, ff, E, k, router_w, records, quant="mxfp4", act="swiglu", router_bias=None,
                 codebooks=None, keep=(), n_shared=0, bias_mode="logit"):
        self.d, self.ff, self.E, self.k = d, ff, E, k
        self.n_shared, self.bias_mode = n_shared, bias_mode
        self.quant, self.act = quant, act
        self.router_w, self.router_bias, self.records, self.codebooks = router_w, router_bias, records, codebooks
        self._keep = list(keep)
        s = LayerStruct()
        s.d, s.ff, s.E, s.k = d, ff, E, k
        s.act, s.quant = ACT[act], QUANT[quant]
        s.router_w = _ptr(router_w)
        s.router_w_dtype = _dt(router_w)
        s.router_bias = _ptr(router_bias)
        s.mxfp4 = MxExperts(_ptr(records), d, ff, E + n_shared)
        cbs = (ctypes.c_void_p * 3)(*([_ptr(c) for c in codebooks] if codebooks is not None else [None] * 3))
        s.rvq3 = RvqExperts(_ptr(records), cbs, d, ff, E + n_shared)
        s.n_shared = n_shared
        s.bias_mode = BIAS_MODE[bias_mode]
        self.struct = s

    def mx_experts(self):
        return MxExperts(_ptr(self.records), self.d, self.ff, self.E + self.n_shared)

    def rvq_experts(self):
        cbs = (ctypes.c_void_p * 3)(*[_ptr(c) for c in self.codebooks])
        return RvqExperts(_ptr(self.records), cbs, self.d, self.ff, self.E + self.n_shared)


# ----------------------------------------------------------------------------- the steps

def moe_route_topk(ctx, x, router_w, bias, k, topk_idx, gates, ws, stream=None):
    T, d = x.shape
    E = router_w.shape[0]
    _check(lib().moe_route_topk(ctx.handle, _ptr(x), _dt(x), _ptr(router_w), _dt(router_w), _ptr(bias), T, d, E, k,
                                _ptr(topk_idx), _ptr(gates), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_route_topk")


def moe_route_topk_ex(ctx, x, router_w, bias, bias_mode, k, topk_idx, gates, ws, stream=None):
    T, d = x.shape
    E = router_w.shape[0]
    _check(lib().moe_route_topk_ex(ctx.handle, _ptr(x), _dt(x), _ptr(router_w), _dt(router_w), _ptr(bias),
                                   BIAS_MODE[bias_mode], T, d, E, k, _ptr(topk_idx), _ptr(gates), _ptr(ws), ws.numel(),
                                   _stream(stream)), "moe_route_topk_ex")


def moe_bucket_tokens(ctx, topk_idx, E, counts, offsets, pair_ids, ws, stream=None):
    T, k = topk_idx.shape
    _check(lib().moe_bucket_tokens(ctx.handle, _ptr(topk_idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(pair_ids),
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_bucket_tokens")


def moe_expert_ffn_mxfp4(ctx, x, k, layer, offsets, pair_ids, y_pairs, ws, stream=None):
    T = x.shape[0]
    ex = layer.mx_experts()
    _check(lib().moe_expert_ffn_mxfp4(ctx.handle, _ptr(x), _dt(x), T, k, ctypes.byref(ex), ACT[layer.act],
                                      _ptr(offsets), _ptr(pair_ids), _ptr(y_pairs), _ptr(ws), ws.numel(),
                                      _stream(stream)), "moe_expert_ffn_mxfp4")


def moe_expert_ffn_mxfp4_static(ctx, x, k, layer, offsets, pair_ids, y_pairs, stream=None):
    """moe_expert_ffn_mxfp4 with the library's static scratch instead of a workspace."""
    T = x.shape[0]
    ex = layer.mx_experts()
    _check(lib().moe_expert_ffn_mxfp4_static(ctx.handle, _ptr(x), _dt(x), T, k, ctypes.byref(ex), ACT[layer.act],
                                             _ptr(offsets), _ptr(pair_ids), _ptr(y_pairs), _stream(stream)),
           "moe_expert_ffn_mxfp4_static")


def expert_ffn_static_max_bytes():
    return int(lib().moe_expert_ffn_mxfp4_static_max_bytes())


def moe_expert_ffn_rvq3(ctx, x, k, layer, offsets, pair_ids, y_pairs, ws, stream=None):
    T = x.shape[0]
    ex = layer.rvq_experts()
    _check(lib().moe_expert_ffn_rvq3(ctx.handle, _ptr(x), _dt(x), T, k, ctypes.byref(ex), ACT[layer.act],
                                     _ptr(offsets), _ptr(pair_ids), _ptr(y_pairs), _ptr(ws), ws.numel(),
                                     _stream(stream)), "moe_expert_ffn_rvq3")


def moe_combine(ctx, x_resid, y_pairs, gates, k, out, stream=None, x_dtype=None):
    T, d = out.shape
    xdt = _dt(x_resid) if x_resid is not None else (MOE_F32 if x_dtype is None else x_dtype)
    _check(lib().moe_combine(ctx.handle, _ptr(x_resid), xdt, _ptr(y_pairs), _ptr(gates), T, k, d, _ptr(out),
                             _dt(out), _stream(stream)), "moe_combine")


def moe_layer_forward(ctx, layer, x, out, ws, topk_idx_out=None, gates_out=None, counts_out=None, stream=None):
    T = x.shape[0]
    _check(lib().moe_layer_forward(ctx.handle, ctypes.byref(layer.struct), _ptr(x), _dt(x), T, _ptr(out), _dt(out),
                                   _ptr(topk_idx_out), _ptr(gates_out), _ptr(counts_out), _ptr(ws), ws.numel(),
                                   _stream(stream)), "moe_layer_forward")


def records_check_ws_bytes(n, record_bytes):
    return int(lib().moe_records_check_ws_bytes(n, record_bytes))


def moe_records_check(ctx, records, n, record_bytes, ws, expected=None, crc_out=None, stream=None):
    """CRC-32 of n device records (records: device int64 tensor of pointers)
    into crc_out (device int32/uint32 [n]); compared with expected when given
    (a mismatch surfaces at ctx.check())."""
    _check(lib().moe_records_check(ctx.handle, _ptr(records), n, record_bytes, _ptr(expected), _ptr(crc_out),
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_records_check")


def moe_stack_forward(ctx, layers, x, out, ws, stream=None):
    T = x.shape[0]
    arr = (LayerStruct * len(layers))(*[l.struct for l in layers])
    _check(lib().moe_stack_forward(ctx.handle, arr, len(layers), _ptr(x), _dt(x), T, _ptr(out), _dt(out), _ptr(ws),
                                   ws.numel(), _stream(stream)), "moe_stack_forward")


def moe_stack_forward_ex(ctx, layers, x, out, ws, topk_trace=None, gates_trace=None, counts_trace=None, stream=None):
    """moe_stack_forward that also writes every layer's routing (device
    tensors, layer after layer: [n_layers][T][k + n_shared] and
    [n_layers][E + n_shared] when all layers have one shape)."""
    T = x.shape[0]
    arr = (LayerStruct * len(layers))(*[l.struct for l in layers])
    _check(lib().moe_stack_forward_ex(ctx.handle, arr, len(layers), _ptr(x), _dt(x), T, _ptr(out), _dt(out),
                                      _ptr(topk_trace), _ptr(gates_trace), _ptr(counts_trace), _ptr(ws), ws.numel(),
                                      _stream(stream)), "moe_stack_forward_ex")


def moe_rvq3_repack(ctx, src_records, dst_records, n, d, ff, stream=None):
    """Row-major RVQ3 records -> position-major (src_records, dst_records:
    device int64 tensors of n record pointers)."""
    _check(lib().moe_rvq3_repack(ctx.handle, _ptr(src_records), _ptr(dst_records), n, d, ff, _stream(stream)),
           "moe_rvq3_repack")


# ----------------------------------------------------------------------------- experts beyond HBM

def tier_plan(heat, has_host, slot_of, n_slots):
    """moe_tier_plan (host only): (new slot of each expert or -1, experts moved)."""
    import numpy as np
    heat = np.ascontiguousarray(heat, dtype=np.float32)
    has = np.ascontiguousarray(has_host, dtype=np.uint8)
    cur = np.ascontiguousarray(slot_of, dtype=np.int32)
    out = np.empty(heat.size, dtype=np.int32)
    n = lib().moe_tier_plan(heat.size, n_slots, heat.ctypes.data, has.ctypes.data, cur.ctypes.data, out.ctypes.data)
    if n < 0:
        raise MoeError(1, "moe_tier_plan")
    return out, n


class Tier:
    """A moe_tier over one layer's bank.  host_bank: page-locked uint8 CPU
    tensor holding E records stride bytes apart (None entries in `present`
    mark experts without a host copy); slots: CUDA uint8 tensor of n_slots x
    stride bytes; records: CUDA int64 tensor [E], the table the layer reads."""

    def __init__(self, ctx, E, record_bytes, stride, host_bank, slots, n_slots, records, direct_host=True,
                 decay=1.0, present=None):
        self.ctx = ctx
        base = host_bank.data_ptr()
        ptrs = [base + e * stride if (present is None or present[e]) else None for e in range(E)]
        self._host_ptrs = (ctypes.c_void_p * E)(*ptrs)
        self._keep = (host_bank, slots, records)
        d = TierDesc()
        d.E, d.record_bytes, d.host_records = E, record_bytes, ctypes.cast(self._host_ptrs, ctypes.c_void_p)
        d.slots, d.n_slots, d.slot_stride = _ptr(slots), n_slots, stride
        d.records, d.direct_host, d.decay = _ptr(records), 1 if direct_host else 0, decay
        self._desc = d
        h = ctypes.c_void_p()
        _check(lib().moe_tier_create(ctx.handle, ctypes.byref(d), ctypes.byref(h)), "moe_tier_create")
        self.handle = h
        self.E = E

    def observe(self, counts, stream=None):
        _check(lib().moe_tier_observe(self.handle, _ptr(counts), _stream(stream)), "moe_tier_observe")

    def rebalance(self, stream=None):
        n = ctypes.c_int(0)
        _check(lib().moe_tier_rebalance(self.handle, _stream(stream), ctypes.byref(n)), "moe_tier_rebalance")
        return n.value

    def pin(self, experts, stream=None):
        import numpy as np
        a = np.ascontiguousarray(experts, dtype=np.int32)
        _check(lib().moe_tier_pin(self.handle, a.ctypes.data if a.size else None, a.size, _stream(stream)),
               "moe_tier_pin")

    def residency(self):
        """(slot of each expert or -1, heat) as numpy arrays."""
        import numpy as np
        slot = np.empty(self.E, dtype=np.int32)
        heat = np.empty(self.E, dtype=np.float32)
        _check(lib().moe_tier_residency(self.handle, slot.ctypes.data, heat.ctypes.data), "moe_tier_residency")
        return slot, heat

    def close(self):
        if getattr(self, "handle", None):
            lib().moe_tier_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------------------------------- latent projections

def moe_project(ctx, x, w, y, resid=None, stream=None):
    """y[t][n] = resid[t][n] + sum_k w[n][k] x[t][k] (x [T][K], w [N][K], y [T][N])."""
    T, K = x.shape
    N = w.shape[0]
    rdt = _dt(resid) if resid is not None else MOE_F32
    _check(lib().moe_project(ctx.handle, _ptr(x), _dt(x), T, K, _ptr(w), _dt(w), N, _ptr(resid), rdt, _ptr(y), _dt(y),
                             _stream(stream)), "moe_project")


def latent_layer_forward_ws_bytes(layer, D, T):
    return int(lib().moe_latent_layer_forward_ws_bytes(ctypes.byref(layer.struct), D, T))


def moe_latent_layer_forward(ctx, layer, w_in, w_out, x, out, ws, latent_out=None, stream=None):
    """The layer in its latent space for hidden-width x [T][D]: out = x + w_out (MoE delta of bf16(w_in x));
    latent_out (int16/bf16 [T][d], optional) receives bf16(w_in x)."""
    T, D = x.shape
    assert _dt(w_in) == _dt(w_out)
    _check(lib().moe_latent_layer_forward(ctx.handle, ctypes.byref(layer.struct), _ptr(w_in), _ptr(w_out), _dt(w_in), D,
                                          _ptr(x), _dt(x), T, _ptr(out), _dt(out), _ptr(latent_out), _ptr(ws),
                                          ws.numel(), _stream(stream)), "moe_latent_layer_forward")
