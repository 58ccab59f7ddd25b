"""The FP8 -> int4 converter step on the GPU (moe_fp8_block_to_int4, through
the C ABI) against the CPU oracle: packed bytes and row scales bit-exact.

Source of the step: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §06
(FP8 block-scale decoding, then the per-row int4 packer) and §02 (fmt e4m3,
128 x 128 weight blocks).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import serving_router_sigmoid_gb300 as m
    torch.cuda.set_device(0)
    return m


def _check(moe, codes, si):
    q4, s = moe.fp8_block_to_int4(codes.cuda(), si.cuda())
    torch.cuda.synchronize()
    rq, rs = oracle.fp8_block_to_int4(codes.numpy(), si.numpy())
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(q4.cpu().numpy(), rq)


@pytest.mark.parametrize("shape", [(2048, 6144), (6144, 2048), (129, 272), (1, 16), (300, 1000), (3, 7),
                                   (5, 8208), (130, 8192)])
def test_checkpoint_like_matrix_byte_exact(moe, shape):
    """Block-scaled E4M3 codes as a checkpoint holds them (GLM gate/up and down
    shapes, partial blocks, rows the 16-byte path does not take)."""
    codes, si = synth.fp8_checkpoint_matrix(*shape, seed=hash(shape) & 0xFFFF)
    codes[0] = 0  # an all-zero row takes the 1e-8 floor
    _check(moe, codes, si)


def test_every_code_and_arbitrary_scales(moe):
    rng = np.random.default_rng(11)
    O, I = 256, 4096
    codes = rng.integers(0, 256, size=(O, I), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x5A  # the NaN codes are outside the contract
    codes[1, :256] = np.arange(256, dtype=np.uint8)
    codes[1, 0x7F], codes[1, 0xFF] = 0, 0
    si = rng.uniform(1e-4, 1e-2, size=(2, 32)).astype(np.float32)
    _check(moe, torch.from_numpy(codes), torch.from_numpy(si))


def test_ties_round_half_to_even(moe):
    """The hand-worked row (7, 1.5, 2.5, -2.5, 0.5, 3.5, -7, 0 at scale_inv
    0.5: w / s hits exact halves) repeated over a full row."""
    base = np.array([0x4E, 0x3C, 0x42, 0xC2, 0x30, 0x46, 0xCE, 0x00], np.uint8)
    codes = np.tile(base, (4, 64))
    si = np.full((1, 4), 0.5, np.float32)
    q4, s = moe.fp8_block_to_int4(torch.from_numpy(codes).cuda(), torch.from_numpy(si).cuda())
    torch.cuda.synchronize()
    assert (s.cpu().numpy() == np.float32(0.5)).all()
    np.testing.assert_array_equal(q4.cpu().numpy(), np.tile(np.array([0xAF, 0x6A, 0xC8, 0x81], np.uint8), (4, 64)))
    _check(moe, torch.from_numpy(codes), torch.from_numpy(si))


def test_unaligned_buffers_take_the_general_path(moe):
    codes, si = synth.fp8_checkpoint_matrix(64, 512, seed=5)
    buf = torch.empty(64 * 512 + 1, dtype=torch.uint8, device="cuda")
    w8 = buf[1:].view(64, 512)
    w8.copy_(codes.cuda())
    qb = torch.empty(64 * 256 + 1, dtype=torch.uint8, device="cuda")
    q4 = qb[1:].view(64, 256)
    s = torch.empty(64, dtype=torch.float32, device="cuda")
    moe.moe_fp8_block_to_int4(w8, si.cuda(), q4, s)
    torch.cuda.synchronize()
    rq, rs = oracle.fp8_block_to_int4(codes.numpy(), si.numpy())
    np.testing.assert_array_equal(q4.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)


def test_argument_errors(moe):
    with pytest.raises(ValueError):
        moe.fp8_block_to_int4(torch.zeros((4, 16), dtype=torch.uint8, device="cuda"),
                              torch.zeros((2, 1), device="cuda"))
    lib = moe.library()
    assert lib.moe_fp8_block_to_int4(None, None, None, None, -1, 16, None) == moe.MOE_ERR_SHAPE
    assert lib.moe_fp8_block_to_int4(None, None, None, None, 0, 16, None) == moe.MOE_OK
    assert lib.moe_fp8_block_to_int4(None, None, None, None, 2, 16, None) == moe.MOE_ERR_INVALID_ARG


def test_near_ties_take_the_exact_quotient(moe):
    """Columns 0..127 hold +-7 at scale_inv 0.5 (row scale s = 0.5); columns
    128..255 hold 1.5, 2.5, -2.5, 0.5, 3.5, -3.5, 0, -1.5 at a scale_inv a few
    ulps away from 0.5, so their quotients w / s sit within a few ulps of
    half-integers (where a product with the reciprocal may round otherwise
    than the packer's division): still byte-exact."""
    nb = 9
    blk0 = np.tile(np.array([0x4E, 0xCE], np.uint8), (nb * 128, 64))
    blk1 = np.tile(np.array([0x3C, 0x42, 0xC2, 0x30, 0x46, 0xC6, 0x00, 0xBC], np.uint8), (nb * 128, 16))
    codes = np.concatenate([blk0, blk1], axis=1)
    si = np.empty((nb, 2), np.float32)
    si[:, 0] = 0.5
    si[:, 1] = (np.float32(0.5) * (1 + (np.arange(nb) - 4) * np.float32(2.0 ** -21))).astype(np.float32)
    rq, _ = oracle.fp8_block_to_int4(codes, si)
    assert len({bytes(rq[128 * j, 64:68]) for j in range(nb)}) > 1  # the near ties round both ways
    _check(moe, torch.from_numpy(codes), torch.from_numpy(si))
