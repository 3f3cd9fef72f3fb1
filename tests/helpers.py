"""Shared helpers of the test suite (GPU runs and oracle comparisons)."""
from __future__ import annotations

import numpy as np

import oracle
from mixture_experts_layer_prefix_gb300 import synth

BF16_TOL = 2e-2   # max normalised error for bf16 outputs and gradients
F32_TOL = 1e-4    # fp32 layer: fp32 accumulation over at most a few thousand terms


def maxnorm_err(got, ref) -> float:
    """max_i |got_i - ref_i| / max_i |ref_i| (0/0 -> 0)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max() if ref.size else 0.0
    num = np.abs(got - ref).max() if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)


def tol_for(dtype_name: str) -> float:
    return F32_TOL if dtype_name == "f32" else BF16_TOL


def np_of(t):
    return t.detach().float().cpu().numpy()


def oracle_layer_for(inp: synth.Inputs, gpu_logits: np.ndarray, tokens=None, nthreads=None):
    """Oracle forward+backward on the same inputs, routed on the GPU's own fp32
    logits (bit-exact routing is defined given identical logits)."""
    s = inp.s
    x, dy = inp.x(), inp.dy()
    logits = np.asarray(gpu_logits, np.float64)
    if tokens is not None:
        x, dy, logits = x[tokens], dy[tokens], logits[tokens]
    return oracle.layer(x, inp.w_r(), inp.w_gate(), inp.w_up(), inp.w_down(), dy, s.k,
                        logits=logits, nthreads=nthreads)
