"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every symbol include/moe.h declares, and its host-only calls behave."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def built():
    from quantized_expert_ffn_score_gb300 import build
    return build.build()


def declared_symbols():
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^MOE_API [^;]*?\b(moe_\w+)\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("moe_route_topk", "moe_bucket_tokens", "moe_expert_ffn_mxfp4", "moe_expert_ffn_rvq3", "moe_combine",
                 "moe_layer_forward"):
        assert name in syms
    from quantized_expert_ffn_score_gb300 import moe
    assert sorted(moe.EXPORTS) == syms


def test_library_exports_every_declared_symbol(built):
    out = subprocess.run(["nm", "-D", "--defined-only", built], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(moe_\w+)$", out, flags=re.M))
    missing = set(declared_symbols()) - exported
    assert not missing, f"not exported: {sorted(missing)}"
    lib = ctypes.CDLL(built)
    for s in declared_symbols():
        assert getattr(lib, s) is not None


def test_host_only_queries(built):
    from quantized_expert_ffn_score_gb300 import moe
    assert moe.mxfp4_record_bytes(3584, 3072) == 17_547_264
    assert moe.rvq3_record_bytes(3584, 3072) == 12_386_304
    assert moe.mxfp4_record_bytes(100, 64) == 0
    assert moe.route_topk_ws_bytes(1, 3584, 896, 16) > 896 * 4
    assert moe.route_topk_ws_bytes(1, 3584, 896, 0) == 0
    assert moe.route_topk_ws_bytes(1, 3584, 10, 16) == 0  # k > E
    assert moe.route_topk_ws_bytes(1, 3584, 4096, 16) == 0  # E above the limit
    assert moe.bucket_tokens_ws_bytes(512, 16, 896) >= 897 * 4
    assert moe.expert_ffn_ws_bytes(512, 16, 3584, 3072, 896) >= 512 * 16 * 3072 * 4
    assert moe.expert_ffn_ws_bytes(8, 16, 3584, 3072, 896, "rvq3") > moe.expert_ffn_ws_bytes(8, 16, 3584, 3072, 896)
    assert moe.expert_ffn_ws_bytes(1, 16, 3584, 8192, 896) == 0  # ff above the limit
    assert "sm_103a" in moe.version()
    # record check: one word per 4 KiB unit of every record
    assert moe.records_check_ws_bytes(896, 17_547_264) >= 896 * 4284 * 4
    assert moe.records_check_ws_bytes(4, 1000) == 0  # not a multiple of 16
    assert moe.records_check_ws_bytes(4, 0) == 0


def test_layer_workspace_covers_shared_experts_and_validates_them(built):
    # host-only: the layer struct's pointers are never dereferenced by the size query
    from quantized_expert_ffn_score_gb300 import moe
    L = moe.lib()

    def ws(n_shared=0, bias_mode=0, bank_E=None, k=16, T=4):
        s = moe.LayerStruct()
        s.d, s.ff, s.E, s.k = 3584, 3072, 896, k
        s.act, s.quant = 0, 0
        s.router_w, s.router_w_dtype = 0x1000, 1
        s.mxfp4 = moe.MxExperts(0x2000, 3584, 3072, 896 + n_shared if bank_E is None else bank_E)
        s.n_shared, s.bias_mode = n_shared, bias_mode
        return L.moe_layer_forward_ws_bytes(ctypes.byref(s), T)

    base, shared = ws(), ws(n_shared=2)
    # two more pairs per token: their h (ff floats) and y (d floats), plus the larger expert tables
    assert shared - base >= 4 * 2 * (3072 + 3584) * 4
    assert ws(n_shared=2, bias_mode=1) == shared
    assert ws(bias_mode=2) == 0                  # unknown bias mode
    assert ws(n_shared=2, bank_E=896) == 0       # the bank must hold the shared records too
    assert ws(n_shared=17) == 0                  # k + n_shared above 32
    assert ws(n_shared=-1) == 0


def test_null_context_is_rejected_without_touching_a_gpu(built):
    from quantized_expert_ffn_score_gb300 import moe
    L = moe.lib()
    rc = L.moe_route_topk(None, None, 0, None, 0, None, 1, 32, 4, 2, None, None, None, 0, None)
    assert rc == 1  # MOE_ERR_INVALID_ARG
    rc = L.moe_layer_forward(None, None, None, 0, 1, None, 0, None, None, None, None, 0, None)
    assert rc == 1
    assert L.moe_status_str(6) == b"a routed expert's record is missing"
    assert L.moe_records_check(None, None, 1, 64, None, None, None, 0, None) == 1
    assert L.moe_route_topk_ex(None, None, 0, None, 0, None, 0, 1, 32, 4, 2, None, None, None, 0, None) == 1
