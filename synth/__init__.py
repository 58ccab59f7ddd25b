"""Seeded synthetic inputs for the routed-MoE layer.

This module draws random tensors with the shapes and value distributions of the
GLM-5.2 MoE layer workloads.  It holds none of the layer's arithmetic (no
quantisation, routing or expert math): both the CPU oracle's tests and the CUDA
path's tests and benchmark take their inputs from here and nothing else is
shared between them.

Distributions (GLM-5.2 layer shape from the model config printed in the
reader.mx article "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型", §02 模型与硬件):
  x      ~ N(0, 1) fp32, one row per token
  Wr     ~ N(0, 0.02) fp32 [E, D]
  bias   ~ U(-0.1, 0.1) fp32 [E], optionally plus a Zipf(s=1.1) skew term
  expert gate/up [I, D], down [D, I] ~ N(0, 0.02) fp32 (packed to int4 by the
         code under test, never here)

Every tensor comes from its own counter-seeded torch.Generator, so any single
expert of any layer can be regenerated alone (the full GLM layer is ~39 GB of
fp32 weights and is never materialised at once).
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field

import torch

# Zipf skew strength for the router bias.  bias_e = U(-0.1, 0.1) - ZIPF_ALPHA *
# 1.1 * ln(rank_e): the expert of rank 1 gets the largest boost.  The value was
# set by tests/golden/calibrate_zipf.py so that, on a 2048-token GLM-shaped draw,
# the hottest expert is selected by ~15% of tokens (top-8 of 256).
ZIPF_ALPHA = 0.014007
ZIPF_S = 1.1


@dataclass(frozen=True)
class LayerCfg:
    name: str
    D: int
    I: int
    E: int
    K: int
    n_shared: int = 1
    T: int = 1
    routed_scale: float = 2.5
    skew: bool = False
    layers: int = 1
    eps: float = 1e-5
    w_std: float = 0.02
    seed: int = 0

    @property
    def S(self) -> int:
        return self.K + self.n_shared


CONFIGS = {
    # tiny MoE layer: hidden 256, moe_intermediate 128, 16 experts top-2, 1 shared, 4 tokens
    "tiny": LayerCfg("tiny", D=256, I=128, E=16, K=2, T=4),
    # GLM-5.2-shaped single MoE layer, decode batch 1
    "glm_decode_b1": LayerCfg("glm_decode_b1", D=6144, I=2048, E=256, K=8, T=1),
    # verify batch: 4 draft tokens x 2 sequences, Zipf-skewed bias
    "glm_verify_b8": LayerCfg("glm_verify_b8", D=6144, I=2048, E=256, K=8, T=8, skew=True),
    # prefill 2048 tokens, Zipf-skewed bias
    "glm_prefill_2048": LayerCfg("glm_prefill_2048", D=6144, I=2048, E=256, K=8, T=2048, skew=True),
    # stack of 8 GLM-shaped layers with RMSNorm + residual; decode batch 1 and 8
    "glm_stack8_b1": LayerCfg("glm_stack8_b1", D=6144, I=2048, E=256, K=8, T=1, layers=8),
    "glm_stack8_b8": LayerCfg("glm_stack8_b8", D=6144, I=2048, E=256, K=8, T=8, layers=8),
}


def seed_of(*parts) -> int:
    """A 63-bit seed from a tuple of labels (stable across machines)."""
    h = hashlib.blake2b(repr(parts).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(*parts))
    return g


def normal(shape, std, device, *parts) -> torch.Tensor:
    g = _gen(device, *parts)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return t.mul_(std) if std != 1.0 else t


def uniform(shape, lo, hi, device, *parts) -> torch.Tensor:
    g = _gen(device, *parts)
    t = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return t.mul_(hi - lo).add_(lo)


def x_rows(cfg: LayerCfg, T: int, device="cpu", stream: str = "x", attempt: int = 0) -> torch.Tensor:
    """Token activations x ~ N(0,1), [T, D]."""
    return normal((T, cfg.D), 1.0, device, cfg.seed, stream, attempt)


def x_row_redraw(cfg: LayerCfg, t: int, attempt: int, device="cpu", stream: str = "x") -> torch.Tensor:
    """A replacement row for token t from its own substream (attempt >= 1)."""
    return normal((cfg.D,), 1.0, device, cfg.seed, stream, "row", t, attempt)


def router_weight(cfg: LayerCfg, layer: int = 0, device="cpu") -> torch.Tensor:
    return normal((cfg.E, cfg.D), cfg.w_std, device, cfg.seed, "Wr", layer)


def zipf_ranks(cfg: LayerCfg, layer: int = 0) -> torch.Tensor:
    """rank[e] in 1..E from a seeded permutation (rank 1 = hottest)."""
    g = _gen("cpu", cfg.seed, "zipf-perm", layer)
    perm = torch.randperm(cfg.E, generator=g)
    rank = torch.empty(cfg.E, dtype=torch.float64)
    rank[perm] = torch.arange(1, cfg.E + 1, dtype=torch.float64)
    return rank


def router_bias(cfg: LayerCfg, layer: int = 0, device="cpu", alpha: float | None = None) -> torch.Tensor:
    b = uniform((cfg.E,), -0.1, 0.1, "cpu", cfg.seed, "bias", layer).double()
    if cfg.skew or alpha is not None:
        a = ZIPF_ALPHA if alpha is None else alpha
        b = b - a * ZIPF_S * torch.log(zipf_ranks(cfg, layer))
    return b.float().to(device)


def expert_fp32(cfg: LayerCfg, e: int, layer: int = 0, device="cpu"):
    """fp32 (gate [I,D], up [I,D], down [D,I]) of expert e; e == E is the shared expert."""
    gate = normal((cfg.I, cfg.D), cfg.w_std, device, cfg.seed, "gate", layer, e)
    up = normal((cfg.I, cfg.D), cfg.w_std, device, cfg.seed, "up", layer, e)
    down = normal((cfg.D, cfg.I), cfg.w_std, device, cfg.seed, "down", layer, e)
    return gate, up, down


def norm_weight(cfg: LayerCfg, device="cpu") -> torch.Tensor:
    """RMSNorm weight of the layer stack: ones (the pages give no values)."""
    return torch.ones(cfg.D, dtype=torch.float32, device=device)


def expert_bytes(cfg: LayerCfg) -> int:
    """Packed int4 bytes + fp32 row scales of one expert (gate, up, down)."""
    gu = cfg.I * ((cfg.D + 1) // 2) + cfg.I * 4
    dn = cfg.D * ((cfg.I + 1) // 2) + cfg.D * 4
    return 2 * gu + dn


def fp8_checkpoint_matrix(O: int, I: int, seed, device="cpu", std: float = 0.02):
    """An FP8 E4M3 weight matrix as a block-scaled checkpoint stores it:
    w ~ N(0, std) fp32, one scale_inv per 128 x 128 block = block amax / 448
    (the largest E4M3 value), codes = w / scale_inv rounded to E4M3 by torch's
    float8_e4m3fn cast.  Returns (codes [O, I] uint8, scale_inv fp32
    [ceil(O/128), ceil(I/128)]).  Input generation only: the converter under
    test decodes these codes, nothing here packs to int4."""
    w = normal((O, I), std, device, "fp8-ckpt", seed)
    bo, bi = (O + 127) // 128, (I + 127) // 128
    pad = torch.zeros((bo * 128, bi * 128), dtype=torch.float32, device=device)
    pad[:O, :I] = w.abs()
    amax = pad.view(bo, 128, bi, 128).amax(dim=(1, 3))
    si = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).float()
    full = si.repeat_interleave(128, 0).repeat_interleave(128, 1)[:O, :I]
    codes = (w / full).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), si.contiguous()
