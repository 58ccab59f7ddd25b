"""The 8-layer GLM-shaped stack (residual MoE blocks, RMSNorm between them)
at decode batch 1 and 8, layer by layer against the oracle.

Every layer's GPU block runs on the GPU's own input (the chain); the oracle
block is applied to that same input, so the comparison of one layer does not
inherit rounding from the layers before it.  A token whose top-K margin at a
layer's normalised input is below the gap the id comparison needs is left out
of that layer's comparison (a near tie may route either way); at least 90% of
the (token, layer) pairs must be compared.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _layers import GAP_MIN, LayerPair

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def moe():
    import serving_router_sigmoid_gb300 as m
    return m


@pytest.mark.parametrize("name", ["glm_stack8_b1", "glm_stack8_b8"])
def test_glm_stack_layerwise_parity(moe, name):
    cfg = synth.CONFIGS[name]
    w = synth.norm_weight(cfg)
    wd = w.cuda()
    x = synth.x_rows(cfg, cfg.T, "cpu", "stack-x")
    xd = x.cuda()
    compared = 0
    for layer in range(cfg.layers):
        pair = LayerPair(cfg, layer=layer, wdev="cuda")
        try:
            x_in = xd.cpu().numpy().copy()
            pair.gpu.moe_block_forward(xd, wd, cfg.eps)
            torch.cuda.synchronize()
            assert pair.gpu.device_status() == 0
            got = xd.cpu().numpy()
            n = np.stack([oracle.rmsnorm(r, w.numpy(), cfg.eps) for r in x_in])
            gap = oracle.router_gap_f64(n, pair.Wr.numpy(), pair.bias.numpy(), cfg.K)
            ok = np.nonzero(gap >= GAP_MIN)[0]
            if len(ok):
                ref = pair.oracle_layer(n[ok]).block_forward(x_in[ok], w.numpy(), cfg.eps)
                d_ref, d_got = ref - x_in[ok], got[ok] - x_in[ok]  # the MoE part of each block
                rel = np.linalg.norm(d_got - d_ref) / np.linalg.norm(d_ref)
                mx = np.abs(d_got - d_ref).max()
                assert rel <= 1e-3, (layer, rel)
                assert mx <= 1e-3 * np.abs(d_ref).max(), (layer, mx)
            compared += len(ok)
        finally:
            pair.close()
            del pair
            torch.cuda.empty_cache()
    assert compared >= 0.9 * cfg.T * cfg.layers
