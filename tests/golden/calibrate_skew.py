"""Calibrates the logit-bias strength of the skewed 128-expert workload.

The skewed 128-expert top-4 layer adds a per-expert logit bias alpha * ln p_e
(p_e proportional to rank^-1.2) so that about 40% of the T*k assignments land
on the 8 busiest experts, with 4 experts pinned empty. This script bisects
alpha with routing computed by the fp64 oracle on the exact seeded inputs and
prints the value stored as SKEW_ALPHA_E128 in the input generator.

Run: python tests/golden/calibrate_skew.py
"""
import dataclasses
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from mixture_experts_layer_prefix_gb300 import synth  # noqa: E402


def top8_share(s, base_logits, alpha):
    inp = synth.Inputs(dataclasses.replace(s, zipf_alpha=alpha), seed=0)
    idx = oracle.topk(base_logits + inp.bias()[None, :].astype(np.float64), s.k)
    counts = np.bincount(idx.ravel(), minlength=s.E)
    return np.sort(counts)[::-1][:8].sum() / idx.size, int((counts == 0).sum())


def main():
    s = synth.CONFIGS["e128_top4_skew"]
    inp = synth.Inputs(s, seed=0)
    base = oracle.router_logits(inp.x(), inp.w_r())
    lo, hi = 0.0, 4.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        share, _ = top8_share(s, base, mid)
        if share < 0.40:
            lo = mid
        else:
            hi = mid
    alpha = round(0.5 * (lo + hi), 4)
    share, empty = top8_share(s, base, alpha)
    print(f"alpha={alpha} top8_share={share:.4f} empty_experts={empty}")


if __name__ == "__main__":
    main()
