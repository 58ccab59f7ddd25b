"""The allocation-free layer forward (moe_layer_forward_static).

Some callers may not allocate device memory at all: a plugin whose host
framework owns every byte of the GPU through its own allocator, a runtime
that plans its memory budget up front, or a decode loop where cudaMalloc (which
can synchronise the device) is not allowed.  For them the library offers one
entry point that takes no handle and allocates nothing; its workspace is a
fixed-size static device array of the library.  It runs the same kernels with
the same launch plan as the handle-based moe_layer_forward, so these tests
call it through the C ABI twice in a row, on the same inputs, and require each
output to equal the handle's bit for bit.  Its device-side flags are read with
moe_layer_static_status.  This file is named to be collected last, and it
builds everything it uses itself, so it passes alone in a fresh process as
well as after the other tests.
"""
import ctypes

import pytest
import torch

import synth
from _layers import LayerPair

STATIC_BYTES = (8 << 20) - 256   # the static workspace after its error word
GLM_MAX_TOKENS = 18              # the largest GLM-5.2 batch that fits in it

CASES = [
    ("tiny", dict(D=256, I=128, E=16, K=2, n_shared=1, T=4)),
    ("tiny-T1", dict(D=256, I=128, E=16, K=2, n_shared=1, T=1)),
    ("tiny-T20", dict(D=256, I=128, E=16, K=2, n_shared=1, T=20)),
    ("ragged-noshared", dict(D=1056, I=96, E=40, K=5, n_shared=0, T=9)),
    ("glm-decode-b1", ("glm_decode_b1", None)),
    ("glm-verify-b8", ("glm_verify_b8", None)),
    ("glm-T18", ("glm_decode_b1", GLM_MAX_TOKENS)),  # the largest GLM batch the workspace holds
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,case", CASES, ids=[c[0] for c in CASES])
def test_static_forward_equals_handle_forward_twice(name, case):
    import serving_router_sigmoid_gb300 as moe
    torch.cuda.set_device(0)
    if isinstance(case, tuple):
        cfg = synth.CONFIGS[case[0]]
        pair = LayerPair(cfg, wdev="cuda", T=case[1])
    else:
        cfg = synth.LayerCfg(name, **case, seed=case["T"] * 7 + case["E"])
        pair = LayerPair(cfg, wdev="cpu")
    try:
        xd = pair.x.cuda()
        ref = pair.gpu.forward(xd)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        table = moe.expert_table_device(pair.gpu_experts, xd.device)
        for _ in range(2):
            out = torch.full_like(xd, float("nan"))
            moe.moe_layer_forward_static(cfg.D, cfg.I, cfg.E, cfg.K, cfg.n_shared, cfg.routed_scale,
                                         pair.Wr_d, pair.bias_d, table, xd, out)
            torch.cuda.synchronize()
            assert torch.equal(out, ref)
        assert moe.static_status() == 0
    finally:
        pair.close()
        torch.cuda.empty_cache()


@pytest.mark.gpu
def test_static_status_reports_and_clears_a_device_flag():
    """A token whose selection scores are all NaN (outside the contract; the
    kernels stay memory-safe and choose experts with weight 0) sets flag 1
    (no finite selection score).  The static entry keeps it until
    moe_layer_static_status reads it, as the handle keeps it until
    moe_layer_device_status does; the read clears it."""
    import serving_router_sigmoid_gb300 as moe
    torch.cuda.set_device(0)
    cfg = synth.LayerCfg("nan", D=256, I=128, E=16, K=2, n_shared=1, T=2, seed=3)
    pair = LayerPair(cfg, wdev="cpu")
    try:
        x = pair.x.clone()
        x[1] = float("nan")
        xd = x.cuda()
        table = moe.expert_table_device(pair.gpu_experts, xd.device)
        assert moe.static_status() == 0
        out = torch.empty_like(xd)
        for _ in range(2):  # the flag collects over calls
            moe.moe_layer_forward_static(cfg.D, cfg.I, cfg.E, cfg.K, cfg.n_shared, cfg.routed_scale,
                                         pair.Wr_d, pair.bias_d, table, xd, out)
        assert moe.static_status() == 1
        assert moe.static_status() == 0
        pair.gpu.forward(xd)
        assert pair.gpu.device_status() == 1
        # a valid batch afterwards: no flag, and the same output on both paths
        xv = pair.x.cuda()
        ref = pair.gpu.forward(xv)
        moe.moe_layer_forward_static(cfg.D, cfg.I, cfg.E, cfg.K, cfg.n_shared, cfg.routed_scale,
                                     pair.Wr_d, pair.bias_d, table, xv, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert moe.static_status() == 0 and pair.gpu.device_status() == 0
    finally:
        pair.close()


def test_static_workspace_limit_for_the_glm_layer():
    """18 GLM-5.2 tokens fit in the static workspace, 19 do not (host-side
    size arithmetic only; no kernel runs)."""
    import serving_router_sigmoid_gb300 as moe
    assert moe.workspace_bytes(6144, 2048, 256, 8, 1, GLM_MAX_TOKENS) <= STATIC_BYTES
    assert moe.workspace_bytes(6144, 2048, 256, 8, 1, GLM_MAX_TOKENS + 1) > STATIC_BYTES


def test_static_forward_rejects_a_batch_beyond_its_workspace():
    """The size check comes before any pointer is used, so placeholder
    pointers never reach a kernel."""
    import serving_router_sigmoid_gb300 as moe
    lib = moe.library()
    dummy = ctypes.c_void_p(16)
    for T in (GLM_MAX_TOKENS + 1, 512):
        desc = moe.MoeLayerDesc(6144, 2048, 256, 8, 1, 2.5, 1)
        rc = lib.moe_layer_forward_static(ctypes.byref(desc), dummy, dummy, dummy, dummy, T, dummy, None)
        assert rc == moe.MOE_ERR_SHAPE
        msg = lib.moe_last_error().decode()
        assert "static workspace" in msg and f"n_tokens={T}" in msg


def test_expert_table_rejects_a_misaligned_weight():
    """The binding checks, on the host, what the entry point cannot check in a
    device table (only the data pointers are read; no kernel runs)."""
    import serving_router_sigmoid_gb300 as moe

    class FakeTensor:
        def __init__(self, p):
            self.p = p
            self.is_cuda = True

        def data_ptr(self):
            return self.p

        def is_contiguous(self):
            return True

    ok = [FakeTensor(4096) for _ in range(6)]
    bad = list(ok)
    bad[2] = FakeTensor(4096 + 8)  # up_q
    with pytest.raises(ValueError, match="up_q must be 16-byte aligned"):
        moe.expert_table_device([ok, bad], "cpu")
    with pytest.raises(ValueError, match="six tensors"):
        moe.expert_table_device([ok[:5]], "cpu")
