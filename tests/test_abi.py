"""The C-ABI library loads without a GPU and exports every symbol its header
declares; host-side argument validation answers before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
HEADER = os.path.join(ROOT, "include", "moe_int4.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import serving_router_sigmoid_gb300 as moe
    return moe.library()


def test_header_declares_the_layer_path_calls():
    names = declared_functions()
    for n in ("moe_pack_int4", "moe_pack_int8", "moe_fp8_block_to_int4", "moe_quant_act_int8",
              "moe_router_topk", "moe_layer_forward", "moe_layer_forward_host", "moe_layer_create",
              "moe_layer_destroy", "moe_block_forward", "moe_layer_debug", "moe_layer_forward_static",
              "moe_layer_static_status", "moe_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_has_no_torch_dependency():
    import serving_router_sigmoid_gb300 as moe
    out = os.popen(f"ldd {moe.LIB_PATH} 2>/dev/null").read()
    assert "torch" not in out and "c10" not in out


def test_host_validation_without_gpu(lib):
    import serving_router_sigmoid_gb300 as moe
    assert lib.moe_pack_int4(None, None, None, -1, 5, None) == moe.MOE_ERR_SHAPE
    assert b"O=-1" in lib.moe_last_error()
    assert lib.moe_pack_int4(None, None, None, 0, 5, None) == moe.MOE_OK  # empty: nothing to do
    assert lib.moe_pack_int4(None, None, None, 3, 5, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_act_int8(None, None, None, 2, 0, None) == moe.MOE_ERR_SHAPE
    assert lib.moe_fp8_block_to_int4(None, None, None, None, -1, 16, None) == moe.MOE_ERR_SHAPE
    assert lib.moe_fp8_block_to_int4(None, None, None, None, 0, 16, None) == moe.MOE_OK
    assert lib.moe_fp8_block_to_int4(None, None, None, None, 2, 16, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_router_topk(None, None, None, 1, 64, 16, 17, 2.5, None, None, None) == moe.MOE_ERR_SHAPE
    for bad in (dict(D=100), dict(I=0), dict(E=0), dict(E=600), dict(K=9, E=8), dict(n_shared=2),
                dict(max_tokens=0)):
        d = dict(D=6144, I=2048, E=256, K=8, n_shared=1, max_tokens=16)
        d.update(bad)
        desc = moe.MoeLayerDesc(d["D"], d["I"], d["E"], d["K"], d["n_shared"], 2.5, d["max_tokens"])
        h = ctypes.c_void_p()
        assert lib.moe_layer_create(ctypes.byref(desc), None, None, None, ctypes.byref(h)) == moe.MOE_ERR_SHAPE, bad
    assert lib.moe_layer_forward(None, None, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_destroy(None) == moe.MOE_OK


def test_workspace_size_glm_decode():
    import serving_router_sigmoid_gb300 as moe
    n1 = moe.workspace_bytes(6144, 2048, 256, 8, 1, 1)
    n2048 = moe.workspace_bytes(6144, 2048, 256, 8, 1, 2048)
    assert n1 < 4 << 20
    # h (fp32), expert outputs (fp32) and the tcgen05 GEMMs' f16 operand rows
    # per (token, slot) dominate: 9 * ((2048 + 6144) * 4 + 6144 * 2) B per token
    assert abs(n2048 - 2048 * 9 * ((2048 + 6144) * 4 + 6144 * 2)) < 0.2 * n2048
