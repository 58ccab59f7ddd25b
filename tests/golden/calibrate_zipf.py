"""Calibrate the Zipf skew strength of the synthetic router bias.

Finds alpha >= 0 such that, with bias_e = U(-0.1,0.1) - alpha*1.1*ln(rank_e), the
hottest expert is selected by 15% of the tokens of a 2048-token GLM-shaped draw
(top-8 of 256).  "15% of assignments" cannot hold literally: with 8 distinct
experts per token one expert receives at most 1/8 of all assignments, so the
share is read as a share of tokens.

The sigmoid probabilities come from the oracle's router (bias 0); the selection
for each candidate alpha is then a plain sort.  Prints the alpha; the constant
ZIPF_ALPHA in synth/__init__.py holds the value this script printed.

    python tests/golden/calibrate_zipf.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(__file__), "..", ".."))
import oracle  # noqa: E402
import synth  # noqa: E402


def hottest_share(p, base_bias, ranks, alpha, K):
    c = p + (base_bias - alpha * synth.ZIPF_S * np.log(ranks)).astype(np.float32)[None, :]
    top = np.argsort(-c, axis=1, kind="stable")[:, :K]
    counts = np.bincount(top.reshape(-1), minlength=p.shape[1])
    return counts.max() / p.shape[0]


def main():
    cfg = synth.CONFIGS["glm_prefill_2048"]
    x = synth.x_rows(cfg, cfg.T).numpy()
    Wr = synth.router_weight(cfg).numpy()
    zero = np.zeros(cfg.E, np.float32)
    _, _, p = oracle.router(x, Wr, zero, cfg.K, cfg.routed_scale)
    base = synth.router_bias(cfg, alpha=0.0).numpy().astype(np.float64)
    ranks = synth.zipf_ranks(cfg).numpy()
    lo, hi = 0.0, 1.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if hottest_share(p, base, ranks, mid, cfg.K) < 0.15:
            lo = mid
        else:
            hi = mid
    alpha = 0.5 * (lo + hi)
    print(f"alpha={alpha:.6f} share={hottest_share(p, base, ranks, alpha, cfg.K):.4f}")


if __name__ == "__main__":
    main()
