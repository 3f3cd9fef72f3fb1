"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns all device memory, or a
loop where cudaMalloc's implicit device synchronisation is not allowed) cannot
pass moe_route a workspace. moe_route_noalloc keeps that scratch in an array
compiled into the library. This file checks, through the C ABI, that it gives
the same results as moe_route on two calls in a row (different inputs each
time, so leftovers of the first call in the shared array cannot leak into the
second), and that shapes beyond the array's size are refused. It is named to
run last, after every other test.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_prefix_gb300 import _native as N
from mixture_experts_layer_prefix_gb300 import build as B
from mixture_experts_layer_prefix_gb300 import layer as L
from mixture_experts_layer_prefix_gb300 import synth

pytestmark = pytest.mark.gpu


def _route_both(s, seed):
    inp = synth.Inputs(s, seed=seed)
    p = L.params_from_inputs(inp, N.MOE_BF16)
    ref = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_BF16)
    got = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_BF16)
    N.moe_route(p.x, p.w_router, p.bias, N.MOE_BF16, s.T, s.d, s.E, s.k, ref.logits, 0, ref.topk_idx,
                ref.gates, ref.counts, ref.offsets, ref.dest_row, ref.src_row, ref.workspace)
    N.moe_route_noalloc(p.x, p.w_router, p.bias, N.MOE_BF16, s.T, s.d, s.E, s.k, got.logits, 0,
                        got.topk_idx, got.gates, got.counts, got.offsets, got.dest_row, got.src_row)
    torch.cuda.synchronize()
    assert N.moe_get_device_error() == 0
    return ref, got


def test_route_noalloc_matches_route_on_two_calls():
    B.build()
    N.load()
    s = synth.MoEShape("noalloc", 3000, 256, 128, 4, 64, "bf16", 0.02, zipf_s=1.2, zipf_alpha=0.5, n_dead=2)
    for seed in (11, 12):
        ref, got = _route_both(s, seed)
        for name in ("topk_idx", "counts", "offsets", "dest_row", "src_row"):
            assert torch.equal(getattr(got, name), getattr(ref, name)), name
        np.testing.assert_allclose(got.logits.cpu().numpy(), ref.logits.cpu().numpy(), rtol=0, atol=1e-6)
        np.testing.assert_allclose(got.gates.cpu().numpy(), ref.gates.cpu().numpy(), rtol=0, atol=2e-6)
        assert int(got.offsets[-1]) == s.T * s.k


def test_route_noalloc_refuses_shapes_beyond_its_scratch():
    B.build()
    lib = N.load()
    fake = 0x100000  # never dereferenced: the size check comes first
    # ceil(T/8) * E = 16384 * 128 > 1,048,576
    assert lib.moe_route_noalloc(fake, fake, None, N.MOE_BF16, 131072, 64, 128, 4, fake, 0, fake, fake,
                                 fake, fake, fake, fake, None) == 4
