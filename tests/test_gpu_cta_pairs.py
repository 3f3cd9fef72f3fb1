"""The weight gradients on CTA pairs (moe_use_cta_pairs(1): 2-CTA clusters,
tcgen05.mma.cta_group::2) against the fp64 oracle (bf16), and against the
MXFP8 oracle for the block-scaled pair kernel (end of the file).

The pair kernel walks 128-row K stages, so the shapes cover experts whose rows
end inside a stage (zeroed tail rows in both CTAs' A halves), experts without
rows (exact zero gradients), M and N that are not multiples of the 256-wide
pair tile (boxes past the edge read zeros, stores are masked), a single
expert, and 1024 experts. The whole layer is checked, so a wrong weight
gradient also shows in no other output it could hide behind.
"""
import pytest
import torch

from mixture_experts_layer_prefix_gb300 import _native as N
from mixture_experts_layer_prefix_gb300 import build as B
from mixture_experts_layer_prefix_gb300 import layer as L
from mixture_experts_layer_prefix_gb300 import synth

from test_gpu_parity import SMALL, _shape, check_layer_against_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    N.load()


PAIR_SHAPES = [s for s in SMALL if s.dtype == "bf16"] + [
    # many pair tiles per expert and several full 128-row stages before the tail
    _shape("bf16_pairs_e32_k4_deep", 4096, 512, 32, 4, 256),
    # 300 rows per expert on average: two full stages and a ragged third
    _shape("bf16_pairs_e8_k2_tail", 1200, 768, 8, 2, 384),
]


def run_layer(s, seed, fused=False):
    inp = synth.Inputs(s, seed=seed)
    p = L.params_from_inputs(inp, N.MOE_BF16)
    b = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_BF16)
    N.moe_use_cta_pairs(1)
    try:
        L.forward(p, b, fused=fused)
        L.backward(p, b, fused=fused)
        torch.cuda.synchronize()
    finally:
        N.moe_use_cta_pairs(0)
    assert N.moe_get_device_error() == 0
    return inp, b


@pytest.mark.parametrize("s", PAIR_SHAPES, ids=lambda s: s.name)
def test_cta_pair_weight_gradients_match_oracle(s):
    inp, b = run_layer(s, seed=3)
    check_layer_against_oracle(inp, b, s)


def test_cta_pairs_in_the_fused_dispatch_backward():
    """moe_dispatch_mlp_bwd with pairs on: its GEMM2 weight gradient runs on
    CTA pairs, its GEMM1 weight gradient still gathers rows on single CTAs."""
    s = _shape("bf16_pairs_fused", 2048, 512, 16, 2, 256)
    inp, b = run_layer(s, seed=4, fused=True)
    check_layer_against_oracle(inp, b, s)


def test_cta_pairs_switch_back_to_single_cta():
    """Turning pairs off again gives the single-CTA kernel's bits."""
    s = _shape("bf16_pairs_switch", 1024, 256, 8, 2, 256)
    inp = synth.Inputs(s, seed=5)
    p = L.params_from_inputs(inp, N.MOE_BF16)
    outs = []
    for pairs in (0, 1, 0):
        b = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_BF16)
        N.moe_use_cta_pairs(pairs)
        try:
            L.forward(p, b)
            L.backward(p, b)
            torch.cuda.synchronize()
        finally:
            N.moe_use_cta_pairs(0)
        outs.append((b.dw_gate.clone(), b.dw_up.clone(), b.dw_down.clone()))
    for a, c in zip(outs[0], outs[2]):
        assert torch.equal(a, c)
    # pairs and single CTAs sum the same products in a different order
    for a, c in zip(outs[0], outs[1]):
        err = (a.float() - c.float()).abs().max() / a.float().abs().max().clamp_min(1e-30)
        assert float(err) < 1e-2


# ----------------------------------------------------------------- MXFP8
# With pairs on, the MXFP8 weight gradients run on 256 x 256 pair tiles
# (block-scaled tcgen05.mma.cta_group::2): each CTA holds its own rows' A
# scales and all 256 columns' B scales. The layer is checked against the
# MXFP8 oracle with the same bound as the single-CTA kernels, on the MXFP8
# shapes (skew with empty experts; f = 384, where the second pair tile's odd
# CTA lies past M) and on one with several pair tiles per expert and
# 128-row stages that end inside an expert.
from test_gpu_mxfp8 import MX_SHAPES  # noqa: E402
from test_gpu_mxfp8 import test_mxfp8_layer_parity as _mx_layer_parity  # noqa: E402

MX_PAIR_SHAPES = MX_SHAPES + [synth.MoEShape("mx_pairs_e8_k2_deep", 1400, 512, 8, 2, 256, "mxfp8", 0.02)]


@pytest.mark.parametrize("s", MX_PAIR_SHAPES, ids=lambda s: s.name)
def test_cta_pair_mxfp8_weight_gradients_match_oracle(s):
    N.moe_use_cta_pairs(1)
    try:
        _mx_layer_parity(s)
    finally:
        N.moe_use_cta_pairs(0)


def test_cta_pairs_mxfp8_switch_back_to_single_cta():
    """Turning pairs off again gives the single-CTA MXFP8 kernel's bits."""
    s = synth.MoEShape("mx_pairs_switch", 1024, 256, 8, 2, 256, "mxfp8", 0.02)
    inp = synth.Inputs(s, seed=7)
    p = L.params_from_inputs(inp, N.MOE_MXFP8)
    outs = []
    for pairs in (0, 1, 0):
        b = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_MXFP8)
        N.moe_use_cta_pairs(pairs)
        try:
            L.forward(p, b)
            L.backward(p, b)
            torch.cuda.synchronize()
        finally:
            N.moe_use_cta_pairs(0)
        assert N.moe_get_device_error() == 0
        outs.append((b.dw_gate.clone(), b.dw_up.clone(), b.dw_down.clone()))
    for a, c in zip(outs[0], outs[2]):
        assert torch.equal(a, c)
    for a, c in zip(outs[0], outs[1]):
        err = (a.float() - c.float()).abs().max() / a.float().abs().max().clamp_min(1e-30)
        assert float(err) < 1e-2
