"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars (stated per check below):
  - int4 packing, int8 activations, expert indices, int32 gate/up/down dot
    products: bit-exact;
  - requantised h: equal except for rare +-1 codes where the device expf and
    the host expf differ in the last ulp (count reported, <= 1e-4 of entries);
  - routing weights: relative 2e-6 (sigmoid of logits summed in another order);
  - layer output: relative L2 <= 1e-3 and max |diff| <= 1e-3 * max |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _layers import LayerPair, assert_output_close, gap_filtered_x, unpack_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import serving_router_sigmoid_gb300 as m
    torch.cuda.set_device(0)
    return m


# ----------------------------------------------------------------- pieces

@pytest.mark.parametrize("shape", [(1, 1), (3, 17), (5, 1001), (64, 6144), (2048, 6144), (6144, 2048)])
def test_pack_int4_byte_exact(moe, shape):
    g = torch.Generator().manual_seed(shape[0] * 7919 + shape[1])
    w = torch.randn(shape, generator=g) * 0.02
    w[0] = 0.0
    if shape[0] > 2:
        w[1, : min(8, shape[1])] = torch.tensor([7, 0.5, 1.5, 2.5, -2.5, -0.5, 3.5, -3.5])[: min(8, shape[1])]
    q4, s = moe.pack_int4(w.cuda())
    rq, rs = oracle.pack_int4(w.numpy())
    np.testing.assert_array_equal(q4.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("shape", [(1, 6144), (7, 256), (3, 1001), (2048, 6144)])
def test_quant_act_bit_exact(moe, shape):
    g = torch.Generator().manual_seed(shape[0] + 31 * shape[1])
    x = torch.randn(shape, generator=g)
    x[0] = 0.0
    if shape[0] > 2:
        x[1] *= 1e-30
        x[2, :5] = torch.tensor([127.0, 0.5, 1.5, 2.5, -2.5])[:5] if shape[1] >= 5 else x[2, :5]
    xd = x.cuda()
    xq = torch.empty(shape, dtype=torch.int8, device="cuda")
    sx = torch.empty(shape[0], dtype=torch.float32, device="cuda")
    moe.moe_quant_act_int8(xd, xq, sx)
    rq, rs = oracle.quant_act(x.numpy())
    np.testing.assert_array_equal(xq.cpu().numpy(), rq)
    np.testing.assert_array_equal(sx.cpu().numpy(), rs)


@pytest.mark.parametrize("T,D,E,K", [(37, 256, 16, 2), (20, 6144, 256, 8), (5, 64, 300, 16), (1, 128, 1, 1)])
def test_router_topk_matches_oracle(moe, T, D, E, K):
    cfg = synth.LayerCfg("r", D=D, I=32, E=E, K=K, T=T, seed=T + D)
    Wr, b = synth.router_weight(cfg), synth.router_bias(cfg)
    x = gap_filtered_x(cfg, T, Wr, b)
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(x.cuda(), Wr.cuda(), b.cuda(), K, 2.5, idx, w)
    ri, rw, _ = oracle.router(x.numpy(), Wr.numpy(), b.numpy(), K, 2.5)
    np.testing.assert_array_equal(idx.cpu().numpy(), ri)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=0)


def test_router_exact_tie_goes_to_lower_index(moe):
    cfg = synth.LayerCfg("tie", D=256, I=32, E=16, K=3, T=9)
    Wr, b = synth.router_weight(cfg), synth.router_bias(cfg)
    Wr[11] = Wr[4]
    b[11] = b[4] = 0.5  # always selected, exactly tied
    x = synth.x_rows(cfg, 9)
    idx = torch.empty((9, 3), dtype=torch.int32, device="cuda")
    w = torch.empty((9, 3), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(x.cuda(), Wr.cuda(), b.cuda(), 3, 2.5, idx, w)
    for row in idx.cpu().numpy().tolist():
        assert row.index(4) < row.index(11)


# ------------------------------------------------------------------ layer

def check_layer(pair, sample=None, x=None):
    """Full debug comparison of one forward; sample = token rows the oracle
    recomputes (all rows when None).  Returns (rel_l2, max_abs, hq_mismatch)."""
    cfg = pair.cfg
    x = pair.x if x is None else x
    T = x.shape[0]
    xd = x.cuda()
    out = torch.empty_like(xd)
    dbg = pair.gpu.moe_layer_debug(xd, out, idx=True, w=True, xq=True, sx=True, gate_acc=True, up_acc=True,
                                   hq=True, sh=True, down_acc=True, union=True)
    torch.cuda.synchronize()
    assert pair.gpu.device_status() == 0
    g = {k: v.cpu().numpy() for k, v in dbg.items()}
    got = out.cpu().numpy()
    tok = np.arange(T) if sample is None else np.asarray(sample)
    xs = x.numpy()[tok]
    OL = pair.oracle_layer(xs)
    ref, od = OL.forward(xs, debug=True)

    # routing.  The set of experts of each token is identical (the inputs keep
    # a margin of >= 1e-5 between the K-th and (K+1)-th score, and with
    # adaptive top-p one around the keff decision).  The selection order is
    # identical except inside runs of consecutive picks whose oracle scores
    # c = sigmoid(logit) + bias lie within 1e-5 of each other: there it
    # follows the last bits of the logits, which the GPU sums in another fp32
    # order, and both orders are correct.  Every per-slot array is compared
    # after mapping each oracle slot to the GPU slot holding the same expert;
    # slots that top-p dropped (id -1, weight 0, at the tail on both sides)
    # have no expert output and are not compared.
    gi, oi = g["idx"][tok], od["idx"]
    np.testing.assert_array_equal(np.sort(gi, 1), np.sort(oi, 1))
    kept = oi >= 0
    np.testing.assert_array_equal(gi >= 0, kept)
    assert (np.diff(kept.astype(np.int8), axis=1) <= 0).all()  # dropped slots form the tail
    _, _, p_or = oracle.router(xs, pair.Wr.numpy(), pair.bias.numpy(), cfg.K, cfg.routed_scale)
    c_or = (p_or + pair.bias.numpy()[None, :]).astype(np.float32)
    c_pick = np.take_along_axis(c_or, np.where(kept, oi, 0).astype(np.int64), 1)
    run = np.concatenate([np.zeros((len(tok), 1), np.int64),
                          np.cumsum(np.abs(np.diff(c_pick, axis=1)) >= 1e-5, axis=1)], axis=1)
    perm = np.empty((len(tok), cfg.S), np.int64)
    for j in range(len(tok)):
        pos = {int(e): k for k, e in enumerate(gi[j]) if e >= 0}
        perm[j, :cfg.K] = [pos[int(e)] if e >= 0 else k for k, e in enumerate(oi[j])]
        # the GPU slot of every pick lies inside the pick's run of near ties
        assert all(run[j, perm[j, k]] == run[j, k] for k in range(cfg.K) if kept[j, k]), (j, gi[j], oi[j])
    if cfg.n_shared:
        perm[:, cfg.K] = cfg.K
    n_swapped = int((perm[:, :cfg.K] != np.arange(cfg.K)[None, :]).any(axis=1).sum())
    valid = np.ones((len(tok), cfg.S), bool)
    valid[:, :cfg.K] = kept

    def by_oracle_slot(a, slots=cfg.S):
        p = perm[:, :slots].reshape(perm.shape[0], slots, *([1] * (a.ndim - 2)))
        return np.take_along_axis(a, p, 1)

    np.testing.assert_allclose(by_oracle_slot(g["w"][tok], cfg.K), od["w"], rtol=2e-6, atol=0)
    # int8 activations bit-exact
    np.testing.assert_array_equal(g["xq"][tok], od["xq"])
    np.testing.assert_array_equal(g["sx"][tok], od["sx"])
    # the union: the distinct routed experts once each, then the shared expert
    nu = int(g["n_union"][0])
    un = g["union_experts"][:nu]
    routed = un[:-1] if cfg.n_shared else un
    assert len(set(routed.tolist())) == len(routed)
    assert set(routed.tolist()) == set(g["idx"][g["idx"] >= 0].tolist())
    if cfg.n_shared:
        assert un[-1] == cfg.E
    if sample is None:
        assert set(routed.tolist()) == set(od["uniq"].tolist())
    # exact int32 dot products (every slot with an expert output)
    np.testing.assert_array_equal(by_oracle_slot(g["gate_acc"][tok])[valid], od["gate_acc"][valid])
    np.testing.assert_array_equal(by_oracle_slot(g["up_acc"][tok])[valid], od["up_acc"][valid])
    hq_g, hq_o = by_oracle_slot(g["hq"][tok])[valid], od["hq"][valid]
    mism = int(np.count_nonzero(hq_g != hq_o))
    assert np.abs(hq_g.astype(np.int32) - hq_o.astype(np.int32)).max() <= 1
    assert mism <= 1e-4 * hq_g.size, f"{mism} of {hq_g.size} hq codes differ"
    np.testing.assert_allclose(by_oracle_slot(g["sh"][tok])[valid], od["sh"][valid], rtol=1e-6, atol=0)
    if n_swapped:
        print(f"{n_swapped} token(s) with near-tied picks in another order")
    # down dots bit-exact against the plain integer dot of the oracle's
    # unpacked down weights with the GPU's own hq, one expert at a time (every
    # (token, slot) row of that expert in one product; the int4 x int8
    # products and all their partial sums are integers far below 2^53, so a
    # float64 matrix product of them is exact whatever its summation order)
    eid = np.empty((len(tok), cfg.S), np.int64)
    eid[:, :cfg.K] = g["idx"][tok]
    if cfg.n_shared:
        eid[:, cfg.K] = cfg.E
    hq_rows, dn_rows = g["hq"][tok], g["down_acc"][tok]
    for e in np.unique(eid[eid >= 0]):
        sel = eid == e
        dq = pair.down_codes(int(e)).astype(np.float64)
        ad = hq_rows[sel].astype(np.float64) @ dq.T
        np.testing.assert_array_equal(dn_rows[sel], ad.astype(np.int64))
    r, m = assert_output_close(got[tok], ref)
    return r, m, mism


SMALL_CASES = [
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=4),    # the tiny config
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=1),
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=16),   # largest fused small-batch path
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=17),   # first multi-kernel path
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=64),   # > 8 rows per expert: several row chunks
    dict(D=1056, I=96, E=40, K=5, n_shared=0, T=9),    # ragged chunk counts, no shared expert
    dict(D=512, I=1024, E=8, K=8, n_shared=1, T=3),    # K = E
    dict(D=512, I=256, E=300, K=16, n_shared=1, T=2),  # E > 256, K = 16
    dict(D=512, I=256, E=300, K=16, n_shared=1, T=20),  # K = 16 above the decode sizes: partial router tiles
    dict(D=1056, I=96, E=40, K=5, n_shared=0, T=24),   # batch > 16 on shapes the grouped tiles skip
    dict(D=512, I=256, E=8, K=2, n_shared=1, T=300),   # several token blocks per expert
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: "D{D}-I{I}-E{E}-K{K}-S{n_shared}-T{T}".format(**c))
def test_layer_parity_small(moe, case):
    cfg = synth.LayerCfg("case", **case, seed=case["T"] * 13 + case["E"])
    pair = LayerPair(cfg, wdev="cpu")
    try:
        r, m, mism = check_layer(pair)
        assert mism == 0
        # the same handle reused at a smaller batch and an empty batch
        if cfg.T > 1:
            check_layer(pair, x=pair.x[:1].clone())
        out = torch.empty((0, cfg.D), device="cuda")
        pair.gpu.moe_layer_forward(torch.empty((0, cfg.D), device="cuda"), out)
    finally:
        pair.close()


TOPP_CASES = [
    (dict(D=256, I=128, E=16, K=4, n_shared=1, T=1), 0.7),     # single decode kernel, one token
    (dict(D=256, I=128, E=16, K=4, n_shared=1, T=4), 0.5),
    (dict(D=256, I=128, E=16, K=4, n_shared=1, T=16), 0.7),
    (dict(D=256, I=128, E=16, K=4, n_shared=1, T=17), 0.7),    # large-batch router, tcgen05 GEMMs
    (dict(D=512, I=256, E=8, K=4, n_shared=1, T=300), 0.6),    # several token blocks per expert
    (dict(D=1056, I=96, E=40, K=5, n_shared=0, T=9), 0.8),     # no shared expert
    (dict(D=1056, I=96, E=40, K=5, n_shared=0, T=24), 0.8),    # untiled shapes above 16 tokens
]


@pytest.mark.parametrize("case,top_p", TOPP_CASES,
                         ids=lambda v: f"p{v}" if isinstance(v, float) else
                         "D{D}-I{I}-E{E}-K{K}-S{n_shared}-T{T}".format(**v))
def test_layer_parity_adaptive_top_p(moe, case, top_p):
    """Adaptive expert top-p: the same kept selections, union, integer dots
    and output as the oracle; fewer union experts than plain top-K; at decode
    sizes the four-kernel plan equals the single kernel bit for bit."""
    cfg = synth.LayerCfg("topp", **case, seed=case["T"] * 17 + case["E"])
    pair = LayerPair(cfg, wdev="cpu", top_p=top_p)
    try:
        check_layer(pair)
        xd = pair.x.cuda()
        d = pair.gpu.moe_layer_debug(xd, idx=True, union=True)
        torch.cuda.synchronize()
        idx = d["idx"].cpu().numpy()
        assert (idx < 0).any(), "top-p dropped nothing: the case does not exercise it"
        if cfg.T <= 16:
            a = pair.gpu.forward(xd)
            pair.gpu.set_option(moe.MOE_OPT_DECODE_SINGLE_KERNEL, 0)
            b = pair.gpu.forward(xd)
            pair.gpu.set_option(moe.MOE_OPT_DECODE_SINGLE_KERNEL, 1)
            torch.cuda.synchronize()
            assert torch.equal(a, b)
        assert pair.gpu.device_status() == 0
    finally:
        pair.close()


@pytest.mark.parametrize("T", [1, 5, 40])
def test_forward_host_equals_forward(moe, T):
    """moe_layer_forward_host (host buffers, copies in and out on the stream)
    gives the device forward's output bit for bit, with pinned and with
    pageable host memory; an empty batch does nothing; a batch beyond
    max_tokens is a SHAPE error."""
    cfg = synth.LayerCfg("host", D=256, I=128, E=16, K=2, n_shared=1, T=T, seed=T + 11)
    pair = LayerPair(cfg, wdev="cpu")
    try:
        xd = pair.x.cuda()
        ref = pair.gpu.forward(xd)
        torch.cuda.synchronize()
        for pinned in (True, False):
            xh = pair.x.clone().contiguous()
            oh = torch.full_like(xh, float("nan"))
            if pinned:
                xh, oh = xh.pin_memory(), oh.pin_memory()
            s = torch.cuda.current_stream()
            pair.gpu.forward_host(xh, oh, s)
            s.synchronize()
            assert torch.equal(oh, ref.cpu()), pinned
        assert pair.gpu.device_status() == 0
        empty = torch.empty((0, cfg.D), dtype=torch.float32)
        pair.gpu.forward_host(empty, empty)
        big = torch.zeros((cfg.T + 1, cfg.D), dtype=torch.float32)
        with pytest.raises(moe.MoeError) as e:
            pair.gpu.forward_host(big, big.clone())
        assert e.value.code == moe.MOE_ERR_SHAPE
    finally:
        pair.close()


def test_layer_forward_is_deterministic(moe):
    cfg = synth.LayerCfg("det", D=256, I=128, E=16, K=2, n_shared=1, T=40, seed=5)
    pair = LayerPair(cfg, wdev="cpu")
    try:
        xd = pair.x.cuda()
        a, b = pair.gpu.forward(xd), pair.gpu.forward(xd)
        torch.cuda.synchronize()
        assert torch.equal(a, b)
    finally:
        pair.close()


def test_block_forward_matches_oracle_block(moe):
    cfg = synth.LayerCfg("blk", D=256, I=128, E=16, K=2, n_shared=1, T=6, seed=9)
    pair = LayerPair(cfg, wdev="cpu")
    try:
        w = synth.norm_weight(cfg)
        x = pair.x * 3.0
        n = np.stack([oracle.rmsnorm(r, w.numpy(), cfg.eps) for r in x.numpy()])
        keep = oracle.router_gap_f64(n, pair.Wr.numpy(), pair.bias.numpy(), cfg.K) >= 1e-5
        assert keep.sum() >= 4
        x, n = x[torch.from_numpy(keep)].contiguous(), n[keep]
        xd = x.cuda().contiguous()
        pair.gpu.moe_block_forward(xd, w.cuda(), cfg.eps)
        torch.cuda.synchronize()
        ref = pair.oracle_layer(n).block_forward(x.numpy(), w.numpy(), cfg.eps)
        assert_output_close(xd.cpu().numpy() - x.numpy(), ref - x.numpy())
    finally:
        pair.close()


def test_layer_rejects_bad_arguments(moe):
    cfg = synth.LayerCfg("bad", D=256, I=128, E=16, K=2, n_shared=1, T=4)
    pair = LayerPair(cfg, wdev="cpu")
    try:
        xd = pair.x.cuda()
        with pytest.raises(moe.MoeError) as ei:
            pair.gpu.moe_layer_forward(torch.zeros((5, cfg.D), device="cuda"), torch.zeros((5, cfg.D), device="cuda"))
        assert ei.value.code == moe.MOE_ERR_SHAPE
        with pytest.raises(ValueError):
            pair.gpu.forward(pair.x)  # host tensor: no CPU path
        with pytest.raises(moe.MoeError) as ei:
            pair.gpu.moe_layer_forward(xd, xd)
        assert ei.value.code == moe.MOE_ERR_INVALID_ARG
    finally:
        pair.close()


# ------------------------------------------------------- GLM-shaped layer

@pytest.mark.slow
@pytest.mark.parametrize("name,top_p", [("glm_decode_b1", 0.0), ("glm_verify_b8", 0.0), ("glm_prefill_2048", 0.0),
                                        ("glm_decode_b1", 0.7), ("glm_verify_b8", 0.7), ("glm_prefill_2048", 0.7)])
def test_glm_layer_parity(moe, name, top_p):
    """The GLM-shaped layer at decode batch 1, verify batch 8 and prefill 2048
    tokens (Zipf-skewed routing: the hottest expert gets ~300 tokens, several
    tcgen05 token blocks), every token compared with the oracle; plain top-8
    and adaptive top-p 0.7."""
    sample = None
    cfg = synth.CONFIGS[name]
    pair = LayerPair(cfg, wdev="cuda", top_p=top_p)
    try:
        # GPU packing of a few full-size experts is byte-exact with the oracle's
        for e in (0, cfg.E):
            gq, gs, uq, us, dq, ds = [t.cpu().numpy() for t in pair.gpu_experts[e]]
            px = pair.oracle_expert(e)
            for a, b in ((gq, px.gq), (gs, px.gs), (uq, px.uq), (us, px.us), (dq, px.dq), (ds, px.ds)):
                np.testing.assert_array_equal(a, b)
        r, m, mism = check_layer(pair, sample)
        print(f"{name} top_p={top_p}: rel_l2={r:.2e} max_abs={m:.2e} hq_mismatch={mism}")
    finally:
        pair.close()
        torch.cuda.empty_cache()
