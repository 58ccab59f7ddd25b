"""The expert GEMMs of batches larger than 16 tokens on the tcgen05 tensor
cores (kind::f16 with the int4 / int8 values carried exactly).

Parity of that path against the oracle is covered by the T > 16 cases of
test_gpu_parity.py, which run it by default.  Here: the tcgen05 and the
legacy integer-MMA plans agree bit for bit (outputs and every int32 dot), and
a saturated layer whose dot products all reach 6144 * 7 * 127 = 5,462,016 is
exact against the oracle (the fp32 accumulator must not lose a unit).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _layers import LayerPair

pytestmark = pytest.mark.gpu

TCGEN05 = 3  # MOE_OPT_TCGEN05_GEMM
TCGEN05_AVAILABLE = 5  # MOE_OPT_TCGEN05_GEMM_AVAILABLE

CASES = [
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=17),
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=64),
    dict(D=512, I=256, E=8, K=2, n_shared=1, T=300),   # 2-3 token blocks per expert
    dict(D=768, I=384, E=32, K=6, n_shared=0, T=129),  # ragged token blocks, no shared expert
]


def _ids(c):
    return "D{D}-I{I}-E{E}-K{K}-S{n_shared}-T{T}".format(**c)


@pytest.fixture(scope="module")
def moe():
    import serving_router_sigmoid_gb300 as m
    return m


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_tcgen05_and_legacy_mma_bit_identical(moe, case):
    cfg = synth.LayerCfg("pf", **case, seed=case["T"] + 3 * case["E"])
    pair = LayerPair(cfg, wdev="cpu")
    try:
        xd = pair.x.cuda()
        assert pair.gpu.get_option(TCGEN05_AVAILABLE) == 1
        want = dict(gate_acc=True, up_acc=True, hq=True, down_acc=True)
        outs, dbgs = [], []
        for opt in (1, 0):
            pair.gpu.set_option(TCGEN05, opt)
            out = torch.empty_like(xd)
            dbgs.append(pair.gpu.moe_layer_debug(xd, out, **want))
            outs.append(out)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        for k in want:
            key = k
            assert torch.equal(dbgs[0][key], dbgs[1][key]), k
        assert torch.equal(outs[0], outs[1])
    finally:
        pair.close()


TMA_WEIGHTS = 6  # MOE_OPT_TCGEN05_TMA_WEIGHTS


@pytest.mark.parametrize("case", CASES + [dict(D=512, I=512, E=64, K=8, n_shared=1, T=2000)], ids=_ids)
def test_tma_and_register_weight_paths_bit_identical(moe, case):
    """The packed weights by TMA (per-expert tensor maps, the default) and by
    the converter threads' register loads (the allocation-free entry point's
    path) give the same int32 dots and outputs; a tile count several times
    the SM count exercises both rings across many tiles per CTA."""
    cfg = synth.LayerCfg("pfw", **case, seed=case["T"] + 5 * case["E"])
    pair = LayerPair(cfg, wdev="cpu")
    try:
        xd = pair.x.cuda()
        assert pair.gpu.get_option(TCGEN05_AVAILABLE) == 1
        assert pair.gpu.get_option(TMA_WEIGHTS) == 1
        want = dict(gate_acc=True, up_acc=True, hq=True, down_acc=True)
        outs, dbgs = [], []
        for opt in (1, 0):
            pair.gpu.set_option(TMA_WEIGHTS, opt)
            assert pair.gpu.get_option(TMA_WEIGHTS) == opt
            out = torch.empty_like(xd)
            dbgs.append(pair.gpu.moe_layer_debug(xd, out, **want))
            outs.append(out)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        for k in want:
            assert torch.equal(dbgs[0][k], dbgs[1][k]), k
        assert torch.equal(outs[0], outs[1])
    finally:
        pair.close()


def test_saturated_dots_exact(moe):
    """All weights +c (int4 code 7) and all activations 1.0 (int8 code 127):
    every gate/up dot is 6144 * 7 * 127 = 5,462,016, near the 2^24 limit of
    exact fp32 accumulation; the down dots are 128 * 7 * 127 per row."""
    D, I, E, K, T = 6144, 128, 4, 2, 24
    dev = torch.device("cuda")
    Wr = torch.zeros((E, D), dtype=torch.float32)
    Wr[0, :] = 1e-3  # expert 0 and 1 always win
    Wr[1, :] = 5e-4
    bias = torch.zeros(E, dtype=torch.float32)
    experts_np, experts_gpu = {}, []
    for e in range(E + 1):
        g = torch.full((I, D), 0.01 * (e + 1), dtype=torch.float32)
        u = torch.full((I, D), -0.02 * (e + 1), dtype=torch.float32)
        d = torch.full((D, I), 0.03 * (e + 1), dtype=torch.float32)
        experts_np[e] = oracle.pack_expert(g.numpy(), u.numpy(), d.numpy())
        gq, gs = moe.pack_int4(g.to(dev))
        uq, us = moe.pack_int4(u.to(dev))
        dq, ds = moe.pack_int4(d.to(dev))
        experts_gpu.append((gq, gs, uq, us, dq, ds))
    x = torch.ones((T, D), dtype=torch.float32)
    layer = moe.MoeLayer(D, I, E, K, 1, 2.5, T, Wr.to(dev), bias.to(dev), experts_gpu)
    try:
        assert layer.get_option(TCGEN05_AVAILABLE) == 1
        out = torch.empty((T, D), device=dev)
        dbg = layer.moe_layer_debug(x.to(dev), out, idx=True, gate_acc=True, up_acc=True, down_acc=True, hq=True)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        OL = oracle.Layer(D, I, E, K, 1, 2.5, Wr.numpy(), bias.numpy(), experts_np)
        ref, od = OL.forward(x.numpy(), debug=True)
        np.testing.assert_array_equal(dbg["idx"].cpu().numpy(), od["idx"])
        ga = dbg["gate_acc"].cpu().numpy()
        assert np.abs(ga).max() == 6144 * 7 * 127
        np.testing.assert_array_equal(ga, od["gate_acc"])
        np.testing.assert_array_equal(dbg["up_acc"].cpu().numpy(), od["up_acc"])
        np.testing.assert_array_equal(dbg["hq"].cpu().numpy(), od["hq"])
        np.testing.assert_array_equal(dbg["down_acc"].cpu().numpy(), od["down_acc"])
        got = out.cpu().numpy()
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= 1e-3
    finally:
        layer.close()
