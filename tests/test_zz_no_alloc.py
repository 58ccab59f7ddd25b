"""The allocation-free layer forward (moe_layer_forward_static).

Some callers may not allocate device memory at all: a plugin whose host
framework owns every byte of the GPU through its own allocator, a runtime
that plans its memory budget up front, or a decode loop where cudaMalloc (which
can synchronise the device) is not allowed.  For them the library offers one
entry point that takes no handle and allocates nothing; its workspace is a
fixed-size static device array of the library.  These tests call it through
the C ABI twice in a row, on the same inputs, and compare each output with the
handle-based moe_layer_forward within the layer-output bar used everywhere
else (relative L2 <= 1e-3, max |diff| <= 1e-3 * max |ref|).  This file is
named to be collected last, and it builds everything it uses itself, so it
passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _layers import LayerPair, assert_output_close

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny", dict(D=256, I=128, E=16, K=2, n_shared=1, T=4)),
    ("tiny-T1", dict(D=256, I=128, E=16, K=2, n_shared=1, T=1)),
    ("tiny-T20", dict(D=256, I=128, E=16, K=2, n_shared=1, T=20)),
    ("ragged-noshared", dict(D=1056, I=96, E=40, K=5, n_shared=0, T=9)),
    ("glm-decode-b1", None),
    ("glm-verify-b8", None),
]


@pytest.mark.parametrize("name,case", CASES, ids=[c[0] for c in CASES])
def test_static_forward_matches_handle_forward_twice(name, case):
    import serving_router_sigmoid_gb300 as moe
    torch.cuda.set_device(0)
    if case is None:
        cfg = synth.CONFIGS["glm_decode_b1" if name == "glm-decode-b1" else "glm_verify_b8"]
        pair = LayerPair(cfg, wdev="cuda")
    else:
        cfg = synth.LayerCfg(name, **case, seed=case["T"] * 7 + case["E"])
        pair = LayerPair(cfg, wdev="cpu")
    try:
        xd = pair.x.cuda()
        ref = pair.gpu.forward(xd)
        torch.cuda.synchronize()
        table = moe.expert_table_device(pair.gpu_experts, xd.device)
        for _ in range(2):
            out = torch.full_like(xd, float("nan"))
            moe.moe_layer_forward_static(cfg.D, cfg.I, cfg.E, cfg.K, cfg.n_shared, cfg.routed_scale,
                                         pair.Wr_d, pair.bias_d, table, xd, out)
            torch.cuda.synchronize()
            assert_output_close(out.cpu().numpy(), ref.cpu().numpy())
    finally:
        pair.close()
        torch.cuda.empty_cache()


def test_static_forward_rejects_a_batch_beyond_its_workspace():
    import serving_router_sigmoid_gb300 as moe
    lib = moe.library()
    desc = moe.MoeLayerDesc(6144, 2048, 256, 8, 1, 2.5, 1)
    dummy = ctypes.c_void_p(16)
    rc = lib.moe_layer_forward_static(ctypes.byref(desc), dummy, dummy, dummy, dummy, 512, dummy, None)
    assert rc == moe.MOE_ERR_SHAPE
    msg = lib.moe_last_error().decode()
    assert "static workspace" in msg and "n_tokens=512" in msg
