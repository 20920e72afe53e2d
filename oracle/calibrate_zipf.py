"""Calibrate the scale of the skewed workload's log-Zipf router bias.

The skewed-load workload asks that router logits get a per-expert bias from log
Zipf(s=1.2) ranks so that roughly a fifth of the experts receive no token.  The
pure log-probability (scale 1) leaves about 30% empty on these inputs, so the
scale ``alpha`` is found by bisection on the seed-0 inputs until 20% +- 1% of
the experts are empty.  Routing is the oracle's; run:

    python -m oracle.calibrate_zipf
"""
from __future__ import annotations

import numpy as np

import oracle
from sparse_moe_layer_router_gb300.synthetic import CONFIGS, as_u16, normal_bf16, zipf_bias


def empty_fraction(x, wr, cfg, alpha):
    bias = zipf_bias(cfg.E, cfg.zipf_s, alpha, cfg.seed).numpy()
    ids, _ = oracle.route(x, wr, cfg.k, bias)
    return 1.0 - len(np.unique(ids)) / cfg.E


def main(target=0.20):
    cfg = CONFIGS["skewed"]
    x = as_u16(normal_bf16((cfg.T, cfg.D), 1.0, cfg.seed, 1))
    wr = as_u16(normal_bf16((cfg.E, cfg.D), 0.02, cfg.seed, 2))
    lo, hi = 0.5, 1.5
    for _ in range(12):
        mid = 0.5 * (lo + hi)
        f = empty_fraction(x, wr, cfg, mid)
        print(f"alpha={mid:.4f} empty={f:.4f}", flush=True)
        if abs(f - target) < 0.005:
            break
        if f > target:
            hi = mid
        else:
            lo = mid
    print(f"calibrated alpha={mid:.4f} empty fraction={f:.4f}")
    return mid, f


if __name__ == "__main__":
    main()
