"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns all device memory, or a
loop where cudaMalloc's implicit device synchronisation is not allowed) cannot
pass moe_route a workspace. moe_route_noalloc keeps that scratch in an array
compiled into the library. These tests check, through the C ABI, that it gives
the same results as moe_route:
  - on two calls in a row with different inputs;
  - at exactly the largest accepted shape (ceil(T/8) * E = 1,048,576 ints),
    followed by a smaller shape, so leftovers of a large call in the shared
    array cannot leak into a later, smaller one;
and that shapes beyond the array are refused.

No test here depends on the order in which pytest runs the files: each one
builds its own inputs and compares against moe_route in the same process, so
it passes alone in a fresh process and after every other test. The file name
sorts last only so that, if it fails, a run stopped at the first failure
(pytest -x) has already run every other test.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_prefix_gb300 import _native as N
from mixture_experts_layer_prefix_gb300 import build as B
from mixture_experts_layer_prefix_gb300 import layer as L
from mixture_experts_layer_prefix_gb300 import synth

pytestmark = pytest.mark.gpu

SCRATCH_INTS = 1 << 20  # the array's size: ceil(T / 8) * E must not exceed it


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    N.load()


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


def _route_logits_in(T, E, k, seed):
    """Both calls on the same given fp32 logits (no router GEMM): cheap at large T."""
    rng = np.random.default_rng(seed)
    logits = torch.from_numpy((rng.standard_normal((T, E)) * 2.0).astype(np.float32)).cuda()
    i32, f32 = torch.int32, torch.float32
    outs = []
    for fn in ("ref", "got"):
        o = dict(topk_idx=torch.empty((T, k), dtype=i32, device="cuda"),
                 gates=torch.empty((T, k), dtype=f32, device="cuda"),
                 counts=torch.empty(E, dtype=i32, device="cuda"),
                 offsets=torch.empty(E + 1, dtype=i32, device="cuda"),
                 dest_row=torch.empty((T, k), dtype=i32, device="cuda"),
                 src_row=torch.empty(T * k, dtype=i32, device="cuda"))
        if fn == "ref":
            ws = torch.empty(N.moe_workspace_size(T, 64, E, k, 64, N.MOE_BF16), dtype=torch.uint8, device="cuda")
            N.moe_route(None, None, None, N.MOE_BF16, T, 64, E, k, logits, N.MOE_ROUTE_LOGITS_IN, o["topk_idx"],
                        o["gates"], o["counts"], o["offsets"], o["dest_row"], o["src_row"], ws)
        else:
            N.moe_route_noalloc(None, None, None, N.MOE_BF16, T, 64, E, k, logits, N.MOE_ROUTE_LOGITS_IN,
                                o["topk_idx"], o["gates"], o["counts"], o["offsets"], o["dest_row"], o["src_row"])
        outs.append(o)
    torch.cuda.synchronize()
    assert N.moe_get_device_error() == 0
    return outs


def _same(ref, got, T, k):
    for name in ("topk_idx", "counts", "offsets", "dest_row", "src_row", "gates"):
        assert torch.equal(got[name], ref[name]), name
    assert int(got["offsets"][-1]) == T * k


def test_route_noalloc_matches_route_on_two_calls():
    s = synth.MoEShape("noalloc", 3000, 256, 128, 4, 64, "bf16", 0.02, zipf_s=1.2, zipf_alpha=0.5, n_dead=2)
    for seed in (11, 12):
        ref, got = _route_both(s, seed)
        for name in ("topk_idx", "counts", "offsets", "dest_row", "src_row"):
            assert torch.equal(getattr(got, name), getattr(ref, name)), name
        np.testing.assert_allclose(got.logits.cpu().numpy(), ref.logits.cpu().numpy(), rtol=0, atol=1e-6)
        np.testing.assert_allclose(got.gates.cpu().numpy(), ref.gates.cpu().numpy(), rtol=0, atol=2e-6)
        assert int(got.offsets[-1]) == s.T * s.k


def test_route_noalloc_at_the_size_limit_then_a_smaller_shape():
    T, E, k = 65536, 128, 4
    assert ((T + 7) // 8) * E == SCRATCH_INTS  # exactly the largest accepted shape
    ref, got = _route_logits_in(T, E, k, seed=21)
    _same(ref, got, T, k)
    # a smaller shape right after: its histograms must not pick up the large call's leftovers
    ref, got = _route_logits_in(1000, 96, 3, seed=22)
    _same(ref, got, 1000, 3)


def test_route_noalloc_refuses_shapes_beyond_its_scratch():
    lib = N.load()
    fake = 0x100000  # never dereferenced: the size check comes first
    # ceil(T/8) * E = 8193 * 128 > 1,048,576: one token past the limit
    assert lib.moe_route_noalloc(fake, fake, None, N.MOE_BF16, 65537, 64, 128, 4, fake, 0, fake, fake,
                                 fake, fake, fake, fake, None) == 4
    assert lib.moe_route_noalloc(fake, fake, None, N.MOE_BF16, 131072, 64, 128, 4, fake, 0, fake, fake,
                                 fake, fake, fake, fake, None) == 4
