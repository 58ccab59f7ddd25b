"""int8-weight experts on the GPU (through the C ABI) against the CPU oracle.

Source: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §05 (quantize_rows:
per-row int8 weights, s = amax/127) and §12 (fmt 1, matmul_q_idot: int8
weights x int8 activations, exact integer dot, then the scales).  Bars as in
test_gpu_parity.py: packed codes and scales bit-exact, expert ids, int8
activations and int32 dots bit-exact, h codes within +-1 at <= 1e-4 of
entries, outputs within relative L2 1e-3 and max |diff| 1e-3 * max |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _layers import LayerPair
from test_gpu_parity import check_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import serving_router_sigmoid_gb300 as m
    torch.cuda.set_device(0)
    return m


@pytest.mark.parametrize("shape", [(1, 1), (3, 17), (5, 1001), (64, 6144), (2048, 6144), (6144, 2048)])
def test_pack_int8_byte_exact(moe, shape):
    g = torch.Generator().manual_seed(shape[0] * 31 + shape[1])
    w = torch.randn(shape, generator=g) * 0.02
    w[0] = 0.0
    if shape[0] > 2 and shape[1] >= 10:
        w[1, :10] = torch.tensor([127.0, 0.5, 1.5, 2.5, -2.5, -127.0, 63.5, 64.5, -0.5, 0.0])
    q8, s = moe.pack_int8(w.cuda())
    rq, rs = oracle.quantize_rows(w.numpy(), 8)
    np.testing.assert_array_equal(q8.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)


CASES = [
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=1),
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=4),
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=16),
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=17),
    dict(D=512, I=256, E=8, K=2, n_shared=1, T=64),
    dict(D=1056, I=96, E=40, K=5, n_shared=0, T=9),
    dict(D=512, I=256, E=300, K=16, n_shared=1, T=2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "D{D}-I{I}-E{E}-K{K}-S{n_shared}-T{T}".format(**c))
def test_int8_layer_parity(moe, case):
    cfg = synth.LayerCfg("i8", **case, seed=case["T"] * 5 + case["E"])
    pair = LayerPair(cfg, wdev="cpu", weight_bits=8)
    try:
        r, m, mism = check_layer(pair)
        assert mism == 0
    finally:
        pair.close()


def test_int8_layer_with_adaptive_top_p(moe):
    cfg = synth.LayerCfg("i8p", D=256, I=128, E=16, K=4, n_shared=1, T=6, seed=77)
    pair = LayerPair(cfg, wdev="cpu", weight_bits=8, top_p=0.6)
    try:
        check_layer(pair)
    finally:
        pair.close()


@pytest.mark.slow
def test_int8_glm_decode_b1_parity(moe):
    """The GLM-shaped layer at decode batch 1 with int8 experts (all 257
    packed on the GPU, 2x the bytes of int4)."""
    cfg = synth.CONFIGS["glm_decode_b1"]
    pair = LayerPair(cfg, wdev="cuda", weight_bits=8)
    try:
        for e in (0, cfg.E):
            gq, gs, uq, us, dq, ds = [t.cpu().numpy() for t in pair.gpu_experts[e]]
            px = pair.oracle_expert(e)
            for a, b in ((gq, px.gq), (gs, px.gs), (dq, px.dq), (ds, px.ds)):
                np.testing.assert_array_equal(a, b)
        r, m, mism = check_layer(pair)
        print(f"glm_decode_b1 int8: rel_l2={r:.2e} max_abs={m:.2e} hq_mismatch={mism}")
    finally:
        pair.close()
        torch.cuda.empty_cache()
