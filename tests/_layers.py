"""Test helpers: seeded layers for the CUDA path and the oracle, built from the
same synthetic fp32 draws (synth) and packed independently by each side."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

GAP_MIN = 1e-5  # selection margin c_(K) - c_(K+1) every test token must have (double twin)


def topp_unambiguous(x_np, Wr, b, K, top_p, routed_scale=2.5):
    """Per token: True when adaptive top-p keeps the same selections under
    fp32 rounding of the logits: the prefix sums on both sides of the keff
    decision lie >= GAP_MIN (relative to the weight sum) from the bound, and
    the picks at keff-1 and keff are not a near tie whose order could flip."""
    if not (0.0 < top_p < 1.0):
        return np.ones(x_np.shape[0], bool)
    idx, w, p = oracle.router(x_np, Wr, b, K, routed_scale)
    keff = oracle.topp_keff(w, top_p)
    ok = np.ones(x_np.shape[0], bool)
    for t in range(x_np.shape[0]):
        tot = float(np.sum(w[t], dtype=np.float64))
        run = np.cumsum(w[t].astype(np.float64))
        bound = top_p * tot
        k = int(keff[t])
        margin = abs(run[k - 1] - bound)
        if k >= 2:
            margin = min(margin, abs(bound - run[k - 2]))
        if k < K:
            c = p[t, idx[t]] + b[idx[t]]
            margin = min(margin, abs(float(c[k - 1]) - float(c[k])) * tot)
        ok[t] = margin >= GAP_MIN * max(tot, 1e-30)
    return ok


def gap_filtered_x(cfg, T, Wr_cpu, bias_cpu, stream="x", max_attempts=64, top_p=0.0):
    """x [T, D] (cpu) where every token's top-K margin is >= GAP_MIN (and,
    with adaptive top-p, whose keff decision is unambiguous).  Tokens that
    fail are redrawn from their own substream (attempt 1, 2, ...)."""
    x = synth.x_rows(cfg, T, "cpu", stream)
    Wr, b = Wr_cpu.numpy(), bias_cpu.numpy()

    def good(rows):
        return (oracle.router_gap_f64(rows, Wr, b, cfg.K) >= GAP_MIN) & \
            topp_unambiguous(rows, Wr, b, cfg.K, top_p, cfg.routed_scale)

    bad = np.nonzero(~good(x.numpy()))[0]
    for t in bad:
        for attempt in range(1, max_attempts):
            row = synth.x_row_redraw(cfg, int(t), attempt, "cpu", stream)
            if good(row.numpy()[None, :])[0]:
                x[t] = row
                break
        else:  # pragma: no cover
            raise RuntimeError(f"token {t}: no draw with a top-K margin >= {GAP_MIN}")
    return x


class LayerPair:
    """A GPU layer (library handle) and the recipe to build its oracle twin."""

    def __init__(self, cfg, layer=0, max_tokens=None, wdev="cuda", x_stream="x", T=None, top_p=0.0,
                 weight_bits=4):
        import serving_router_sigmoid_gb300 as moe
        self.cfg, self.layer, self.wdev, self.top_p = cfg, layer, wdev, float(top_p)
        self.weight_bits = int(weight_bits)
        pack = moe.pack_int4 if self.weight_bits == 4 else moe.pack_int8
        dev = torch.device("cuda")
        self.Wr = synth.router_weight(cfg, layer)
        self.bias = synth.router_bias(cfg, layer)
        T = cfg.T if T is None else T
        self.x = gap_filtered_x(cfg, T, self.Wr, self.bias, x_stream, top_p=self.top_p)
        self.gpu_experts = []
        for e in range(cfg.E + cfg.n_shared):
            g, u, d = synth.expert_fp32(cfg, e, layer, wdev)
            g, u, d = g.to(dev), u.to(dev), d.to(dev)
            gq, gs = pack(g)
            uq, us = pack(u)
            dq, ds = pack(d)
            self.gpu_experts.append((gq, gs, uq, us, dq, ds))
            del g, u, d
        torch.cuda.synchronize()
        self.Wr_d, self.bias_d = self.Wr.to(dev), self.bias.to(dev)
        self.gpu = moe.MoeLayer(cfg.D, cfg.I, cfg.E, cfg.K, cfg.n_shared, cfg.routed_scale,
                                max_tokens or max(T, 1), self.Wr_d, self.bias_d, self.gpu_experts, self.top_p,
                                self.weight_bits)
        self._orc_cache = {}

    def oracle_expert(self, e):
        if e not in self._orc_cache:
            g, u, d = synth.expert_fp32(self.cfg, e, self.layer, self.wdev)
            self._orc_cache[e] = oracle.pack_expert(g.cpu().numpy(), u.cpu().numpy(), d.cpu().numpy(),
                                                    bits=self.weight_bits)
        return self._orc_cache[e]

    def oracle_layer(self, x_np):
        """Oracle layer holding exactly the experts the oracle's own router picks for x."""
        cfg = self.cfg
        idx, _, _ = oracle.router(x_np, self.Wr.numpy(), self.bias.numpy(), cfg.K, cfg.routed_scale)
        need = sorted(set(idx.reshape(-1).tolist()) | ({cfg.E} if cfg.n_shared else set()))
        experts = {e: self.oracle_expert(e) for e in need}
        return oracle.Layer(cfg.D, cfg.I, cfg.E, cfg.K, cfg.n_shared, cfg.routed_scale,
                            self.Wr.numpy(), self.bias.numpy(), experts, top_p=self.top_p,
                            weight_bits=self.weight_bits)

    def down_codes(self, e):
        """The oracle's down weights of expert e as integers [D, I]."""
        px = self.oracle_expert(e)
        return px.dq.astype(np.int64) if self.weight_bits == 8 else unpack_np(px.dq, self.cfg.I)

    def close(self):
        self.gpu.close()


def unpack_np(q4, I):
    lo = (q4 & 15).astype(np.int64) - 8
    hi = (q4 >> 4).astype(np.int64) - 8
    v = np.empty(q4.shape[:-1] + (2 * q4.shape[-1],), np.int64)
    v[..., 0::2], v[..., 1::2] = lo, hi
    return v[..., :I]


def rel_l2(a, b):
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-30))


def assert_output_close(got, ref, rel=1e-3, abs_frac=1e-3):
    """The layer-output bar: relative L2 <= 1e-3 and max|diff| <= 1e-3 * max|ref|."""
    r = rel_l2(got, ref)
    m = float(np.abs(got - ref).max()) if got.size else 0.0
    lim = abs_frac * float(np.abs(ref).max()) if ref.size else 0.0
    assert r <= rel, f"rel L2 {r:.3e} > {rel}"
    assert m <= lim, f"max abs {m:.3e} > {lim:.3e}"
    return r, m
