"""The persistent single-kernel decode layer (batches of 1..16 tokens).

Parity of that kernel against the oracle is covered by the T <= 16 cases of
test_gpu_parity.py, which run it by default.  Here: the four-kernel launch
plan of the same batches against the oracle, the two plans bit-identical to
each other, repeated launches (the kernel's arrival counters must be back at
zero after every launch), CUDA-graph replay, and a batch at every token count
the kernel covers.
"""
import time

import pytest
import torch

import synth
from _layers import LayerPair
from test_gpu_parity import check_layer

pytestmark = pytest.mark.gpu

SINGLE = 1  # MOE_OPT_DECODE_SINGLE_KERNEL
AVAILABLE = 2  # MOE_OPT_DECODE_SINGLE_KERNEL_AVAILABLE
TEST_WAIT_TIMEOUT = 4  # MOE_OPT_DECODE_TEST_WAIT_TIMEOUT
SYNC_TIMEOUT = 16  # error bit of a wait that ran out of time

DECODE_CASES = [
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=1),
    dict(D=256, I=128, E=16, K=2, n_shared=1, T=16),
    dict(D=1056, I=96, E=40, K=5, n_shared=0, T=9),
    dict(D=512, I=1024, E=8, K=8, n_shared=1, T=3),
    dict(D=512, I=256, E=300, K=16, n_shared=1, T=2),
]


def _ids(c):
    return "D{D}-I{I}-E{E}-K{K}-S{n_shared}-T{T}".format(**c)


@pytest.fixture(scope="module")
def moe():
    import serving_router_sigmoid_gb300 as m
    return m


def _pair(case, seed_extra=0):
    cfg = synth.LayerCfg("dec", **case, seed=case["T"] * 7 + case["E"] + seed_extra)
    return LayerPair(cfg, wdev="cpu")


@pytest.mark.parametrize("case", DECODE_CASES, ids=_ids)
def test_single_kernel_is_available(moe, case):
    pair = _pair(case)
    try:
        assert pair.gpu.get_option(AVAILABLE) == 1
        assert pair.gpu.get_option(SINGLE) == 1
    finally:
        pair.close()


@pytest.mark.parametrize("case", DECODE_CASES, ids=_ids)
def test_four_kernel_plan_parity(moe, case):
    pair = _pair(case)
    try:
        pair.gpu.set_option(SINGLE, 0)
        _, _, mism = check_layer(pair)
        assert mism == 0
    finally:
        pair.close()


@pytest.mark.parametrize("case", DECODE_CASES, ids=_ids)
def test_plans_bit_identical(moe, case):
    pair = _pair(case, 1)
    try:
        xd = pair.x.cuda()
        a = pair.gpu.forward(xd)
        pair.gpu.set_option(SINGLE, 0)
        b = pair.gpu.forward(xd)
        pair.gpu.set_option(SINGLE, 1)
        c = pair.gpu.forward(xd)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        assert torch.equal(a, b)
        assert torch.equal(a, c)
    finally:
        pair.close()


def test_every_token_count(moe):
    """One handle, batches of 1..16 tokens (every kernel variant), each equal
    to the four-kernel plan on the same rows."""
    case = dict(D=256, I=128, E=16, K=2, n_shared=1, T=16)
    pair = _pair(case, 2)
    try:
        xd = pair.x.cuda()
        for T in range(1, 17):
            pair.gpu.set_option(SINGLE, 1)
            a = pair.gpu.forward(xd[:T].contiguous())
            pair.gpu.set_option(SINGLE, 0)
            b = pair.gpu.forward(xd[:T].contiguous())
            torch.cuda.synchronize()
            assert torch.equal(a, b), T
        assert pair.gpu.device_status() == 0
    finally:
        pair.close()


def test_repeated_launches_and_graph(moe):
    """200 launches in a row and 50 graph replays give the first output bit
    for bit and leave no error flag (counters cleared by every launch)."""
    case = dict(D=512, I=256, E=64, K=6, n_shared=1, T=5)
    pair = _pair(case, 3)
    try:
        xd = pair.x.cuda()
        ref = pair.gpu.forward(xd)
        out = torch.empty_like(xd)
        for _ in range(200):
            pair.gpu.moe_layer_forward(xd, out)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        assert torch.equal(out, ref)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        out2 = torch.zeros_like(xd)
        with torch.cuda.stream(s):
            pair.gpu.moe_layer_forward(xd, out2, stream=s)  # warm-up outside capture
            s.synchronize()
            with torch.cuda.graph(g, stream=s):
                pair.gpu.moe_layer_forward(xd, out2, stream=s)
        for _ in range(50):
            out2.zero_()
            g.replay()
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        assert torch.equal(out2, ref)
    finally:
        pair.close()


def test_block_forward_single_kernel(moe):
    """The residual block (out aliases the residual) through the single
    kernel equals the four-kernel plan."""
    case = dict(D=256, I=128, E=16, K=2, n_shared=1, T=4)
    pair = _pair(case, 4)
    try:
        w = synth.norm_weight(pair.cfg, "cuda")
        x0 = pair.x.cuda()
        a = x0.clone()
        pair.gpu.moe_block_forward(a, w, 1e-5)
        pair.gpu.set_option(SINGLE, 0)
        b = x0.clone()
        pair.gpu.moe_block_forward(b, w, 1e-5)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        assert torch.equal(a, b)
    finally:
        pair.close()


def test_bad_option_rejected(moe):
    pair = _pair(DECODE_CASES[0])
    try:
        with pytest.raises(moe.MoeError):
            pair.gpu.set_option(SINGLE, 2)
        with pytest.raises(moe.MoeError):
            pair.gpu.set_option(99, 1)
        with pytest.raises(moe.MoeError):
            pair.gpu.get_option(99)
    finally:
        pair.close()


@pytest.mark.parametrize("single", [1, 0])
def test_layer_exact_tie_goes_to_lower_index(moe, single):
    """Two experts with identical router rows and bias always tie exactly;
    the layer's top-K (both launch plans) puts the lower index first and
    matches the oracle's router on the same weights."""
    import oracle
    case = dict(D=256, I=128, E=16, K=3, n_shared=1, T=9)
    pair = _pair(case, 5)
    try:
        pair.gpu.set_option(SINGLE, single)
        # the handle borrows these device tensors
        pair.Wr_d[11] = pair.Wr_d[4]
        pair.bias_d[11] = 0.5
        pair.bias_d[4] = 0.5
        Wr, b = pair.Wr_d.cpu(), pair.bias_d.cpu()
        x = synth.x_rows(pair.cfg, 9)
        dbg = pair.gpu.moe_layer_debug(x.cuda(), idx=True, w=True)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        idx = dbg["idx"].cpu().numpy()
        for row in idx.tolist():
            assert row.index(4) < row.index(11)
        ri, rw, _ = oracle.router(x.numpy(), Wr.numpy(), b.numpy(), 3, pair.cfg.routed_scale)
        assert (idx == ri).all()
    finally:
        pair.close()


@pytest.mark.parametrize("T", [1, 3])
def test_wait_timeout_is_reported_and_recovered(moe, T):
    """The test hook makes the grid barrier's bounded wait run out (it waits
    for one arrival more than there are CTAs): the launch ends after about a
    second with the time-out bit, which device_status reports, and the full
    result; the next launches run normally.  No fault, trap or endless loop
    is involved."""
    case = dict(D=256, I=128, E=16, K=2, n_shared=1, T=T)
    pair = _pair(case, 6)
    try:
        xd = pair.x.cuda()
        ref = pair.gpu.forward(xd)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        pair.gpu.set_option(TEST_WAIT_TIMEOUT, 1)
        assert pair.gpu.get_option(TEST_WAIT_TIMEOUT) == 1
        t0 = time.time()
        out = pair.gpu.forward(xd)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        assert pair.gpu.device_status() == SYNC_TIMEOUT
        assert elapsed > 0.5
        assert torch.equal(out, ref)
        pair.gpu.set_option(TEST_WAIT_TIMEOUT, 0)
        for _ in range(3):
            out2 = pair.gpu.forward(xd)
        torch.cuda.synchronize()
        assert pair.gpu.device_status() == 0
        assert torch.equal(out2, ref)
    finally:
        pair.close()
