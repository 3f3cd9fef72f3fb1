"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Routing metadata must be bit-exact given the GPU's own fp32 logits; float
outputs and gradients must be within the max normalised error of the dtype
(2e-2 for bf16, 1e-4 for the fp32 layer). Shapes span several tiles, ragged
tails, empty experts, and the degenerate cases of the method.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_prefix_gb300 import _native as N
from mixture_experts_layer_prefix_gb300 import build as B
from mixture_experts_layer_prefix_gb300 import layer as L
from mixture_experts_layer_prefix_gb300 import synth

from helpers import maxnorm_err, np_of, oracle_layer_for, tol_for

pytestmark = pytest.mark.gpu

DT = {"f32": N.MOE_F32, "bf16": N.MOE_BF16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    N.load()


def _shape(name, T, d, E, k, f, dtype="bf16", **kw):
    return synth.MoEShape(name, T, d, E, k, f, dtype, kw.pop("router_std", 0.02), **kw)


SMALL = [
    synth.CONFIGS["tiny_fp32"],
    _shape("bf16_e8_k2", 512, 256, 8, 2, 256),
    _shape("bf16_e16_k4_ragged", 1000, 256, 16, 4, 192),
    _shape("bf16_e128_k4", 2048, 256, 128, 4, 128),
    _shape("bf16_skew_dead", 1500, 320, 32, 4, 256, zipf_s=1.2, zipf_alpha=0.8, n_dead=3),
    _shape("bf16_e64_k8", 700, 128, 64, 8, 128, zipf_s=1.0),
    _shape("bf16_single_expert", 300, 128, 1, 1, 128),
    _shape("bf16_k_eq_E", 77, 192, 3, 3, 64),
    _shape("bf16_one_token", 1, 64, 4, 2, 64),
    _shape("bf16_e320_k2", 600, 128, 320, 2, 64),
    # the largest supported expert count: most experts empty, one block ranks all 1024 for the wgrads
    _shape("bf16_e1024_k2", 700, 128, 1024, 2, 64),
]


def run_gpu(s, seed=0):
    dt = DT[s.dtype]
    inp = synth.Inputs(s, seed=seed)
    p = L.params_from_inputs(inp, dt)
    b = L.Buffers(s.T, s.d, s.E, s.k, s.f, dt)
    L.forward(p, b)
    L.backward(p, b)
    torch.cuda.synchronize()
    assert N.moe_get_device_error() == 0
    return inp, p, b


def check_routing(b, s, gpu_logits):
    ref = oracle.route(gpu_logits.astype(np.float64), s.k, s.E)
    np.testing.assert_array_equal(b.topk_idx.cpu().numpy(), ref["topk_idx"])
    np.testing.assert_array_equal(b.counts.cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(b.offsets.cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(b.dest_row.cpu().numpy(), ref["dest_row"])
    np.testing.assert_array_equal(b.src_row.cpu().numpy(), ref["src_row"])
    np.testing.assert_allclose(b.gates.cpu().numpy(), ref["gates"], rtol=0, atol=2e-6)
    return ref


@pytest.mark.parametrize("s", SMALL, ids=lambda s: s.name)
def test_layer_parity(s):
    inp, p, b = run_gpu(s)
    check_layer_against_oracle(inp, b, s)


def check_layer_against_oracle(inp, b, s):
    """Every output of a forward+backward in `b` against the fp64 oracle run on the
    GPU's own logits: routing bit-exact, values within the dtype's tolerance,
    exact zeros for the weight gradients of experts without rows."""
    gl = b.logits.cpu().numpy()
    # router GEMM: fp32 accumulation of exact products vs fp64
    ref_logits = oracle.router_logits(inp.x(), inp.w_r(), inp.bias())
    assert maxnorm_err(gl, ref_logits) < 1e-5
    check_routing(b, s, gl)
    ref = oracle_layer_for(inp, gl)
    tol = tol_for(s.dtype)
    dest = b.dest_row.cpu().numpy().ravel()  # pair p -> row
    f = s.f
    h = np_of(b.h_save)[dest]
    errs = {
        "h_gate": maxnorm_err(h[:, :f], ref["hg"]),
        "h_up": maxnorm_err(h[:, f:], ref["hu"]),
        "a": maxnorm_err(np_of(b.a_save)[dest], ref["a"]),
        "y_perm": maxnorm_err(np_of(b.y_perm)[dest], ref["ye"]),
        "y": maxnorm_err(np_of(b.y), ref["y"]),
        "dy_perm": maxnorm_err(np_of(b.dy_perm)[dest], ref["dye"]),
        "dgates": maxnorm_err(np_of(b.dgates), ref["dgates"]),
        "dlogits": maxnorm_err(np_of(b.dlogits), ref["dlogits"]),
        "dw_router": maxnorm_err(np_of(b.dw_router), ref["dw_r"].T),
        "dw_gate": maxnorm_err(np_of(b.dw_gate), ref["dw_gate"]),
        "dw_up": maxnorm_err(np_of(b.dw_up), ref["dw_up"]),
        "dw_down": maxnorm_err(np_of(b.dw_down), ref["dw_down"]),
        "dx": maxnorm_err(np_of(b.dx), ref["dx"]),
    }
    bad = {k_: v for k_, v in errs.items() if not v <= tol}
    assert not bad, f"{s.name}: {bad} (all: {errs})"
    # experts with no rows get exactly zero weight gradients
    empty = np.flatnonzero(b.counts.cpu().numpy() == 0)
    for e in empty:
        assert float(b.dw_gate[e].abs().max()) == 0.0
        assert float(b.dw_down[e].abs().max()) == 0.0
        assert float(b.dw_router[e].abs().max()) == 0.0


def test_routing_ties_bit_exact_with_given_logits():
    """Logits on a coarse grid (many exact ties, +-0) through MOE_ROUTE_LOGITS_IN."""
    T, E, k = 3000, 40, 5
    rng = np.random.default_rng(0)
    l = (np.round(rng.standard_normal((T, E)) * 2) / 2).astype(np.float32)
    l[::7, :] = 0.0
    l[::11, ::2] = -0.0
    b = L.Buffers(T, 64, E, k, 64, N.MOE_BF16)
    b.logits.copy_(torch.from_numpy(l))
    N.moe_route(None, None, None, N.MOE_BF16, T, 64, E, k, b.logits, N.MOE_ROUTE_LOGITS_IN, b.topk_idx,
                b.gates, b.counts, b.offsets, b.dest_row, b.src_row, b.workspace)
    torch.cuda.synchronize()
    check_routing(b, dataclasses.replace(synth.CONFIGS["e128_top4"], T=T, E=E, k=k), l)


def test_deterministic_bitwise():
    s = _shape("det", 1024, 256, 16, 4, 128)
    _, _, b1 = run_gpu(s)
    outs1 = [t.clone() for t in (b1.y, b1.dx, b1.dw_gate, b1.dw_up, b1.dw_down, b1.dw_router, b1.dest_row)]
    _, _, b2 = run_gpu(s)
    outs2 = (b2.y, b2.dx, b2.dw_gate, b2.dw_up, b2.dw_down, b2.dw_router, b2.dest_row)
    for a, c in zip(outs1, outs2):
        assert torch.equal(a, c)


def test_permute_is_exact_copy():
    s = _shape("perm", 999, 512, 32, 4, 64)
    inp, p, b = run_gpu(s)
    N.moe_permute(p.x, N.MOE_BF16, s.T, s.d, s.k, b.dest_row, b.x_perm)
    torch.cuda.synchronize()
    x = p.x.cpu()
    src = b.src_row.cpu().long() // s.k
    assert torch.equal(b.x_perm.cpu(), x[src])


FUSED_SHAPES = [
    _shape("fused_ragged", 1000, 256, 16, 4, 192),
    _shape("fused_skew_dead", 1500, 320, 32, 4, 256, zipf_s=1.2, zipf_alpha=0.8, n_dead=3),
    _shape("fused_e320_k2", 600, 128, 320, 2, 64),
    _shape("fused_one_token", 1, 64, 4, 2, 64),
    _shape("fused_e8_k2_wide", 2048, 1024, 8, 2, 512),
]


@pytest.mark.parametrize("s", FUSED_SHAPES, ids=lambda s: s.name)
def test_fused_dispatch_matches_oracle_and_permute_path(s):
    """The dispatch fused into GEMM1 and its weight gradient (rows gathered from
    x through src_row): every output against the fp64 oracle, and bit-identical
    to moe_permute + the grouped MLP (both read the same values)."""
    dt = N.MOE_BF16
    inp = synth.Inputs(s, seed=2)
    p = L.params_from_inputs(inp, dt)
    outs = []
    for fused in (False, True):
        b = L.Buffers(s.T, s.d, s.E, s.k, s.f, dt)
        L.forward(p, b, fused=fused)
        L.backward(p, b, fused=fused)
        torch.cuda.synchronize()
        assert N.moe_get_device_error() == 0
        if fused:
            check_layer_against_oracle(inp, b, s)
        outs.append([t.clone() for t in (b.h_save, b.a_save, b.y_perm, b.y, b.dx_perm, b.dx, b.dw_gate, b.dw_up,
                                         b.dw_down, b.dw_router)])
    names = ("h_save", "a_save", "y_perm", "y", "dx_perm", "dx", "dw_gate", "dw_up", "dw_down", "dw_router")
    for n_, a, c in zip(names, *outs):
        assert torch.equal(a, c), n_


def test_fused_dispatch_rejects_other_dtypes():
    b = L.Buffers(8, 64, 4, 2, 64, N.MOE_F32)
    w = torch.zeros(4, 64, 64, device="cuda")
    with pytest.raises(N.MoEError):
        N.moe_dispatch_mlp_fwd(torch.zeros(8, 64, device="cuda"), b.src_row, 8, 2, w, w, w, N.MOE_F32, b.offsets,
                               4, 64, 64, b.h_save, b.a_save, b.y_perm)


def test_zero_tokens():
    b = L.Buffers(0, 64, 8, 2, 64, N.MOE_BF16)
    p = L.Params(x=torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"),
                 w_router=torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda"), bias=None,
                 w_gate=torch.zeros(8, 64, 64, dtype=torch.bfloat16, device="cuda"),
                 w_up=torch.zeros(8, 64, 64, dtype=torch.bfloat16, device="cuda"),
                 w_down=torch.zeros(8, 64, 64, dtype=torch.bfloat16, device="cuda"),
                 dy=torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"))
    L.forward(p, b)
    L.backward(p, b)
    torch.cuda.synchronize()
    assert N.moe_get_device_error() == 0
    assert torch.all(b.counts == 0) and torch.all(b.offsets == 0)
    assert float(b.dw_gate.float().abs().max()) == 0.0


def test_host_pipeline_matches_direct_calls():
    """The copy-overlapped host pipeline gives, step by step, the same bits as
    calling forward and backward directly on the same batches (the layer is
    deterministic), including the router weight gradient of the last step."""
    s = _shape("bf16_pipe", 1000, 256, 16, 4, 192)
    dt = N.MOE_BF16
    inp = synth.Inputs(s, seed=3)
    p = L.params_from_inputs(inp, dt)
    b = L.Buffers(s.T, s.d, s.E, s.k, s.f, dt)
    g = torch.Generator().manual_seed(11)
    xs = [torch.randn(s.T, s.d, generator=g).to(torch.bfloat16).pin_memory() for _ in range(3)]
    dys = [torch.randn(s.T, s.d, generator=g).to(torch.bfloat16).pin_memory() for _ in range(3)]
    ys = [torch.empty(s.T, s.d, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    dxs = [torch.empty_like(y).pin_memory() for y in ys]
    L.HostPipeline(p, b).run(xs, dys, ys, dxs)
    torch.cuda.synchronize()
    assert N.moe_get_device_error() == 0
    dwr_pipe = b.dw_router.clone()
    for i in range(3):
        p.x.copy_(xs[i])
        p.dy.copy_(dys[i])
        L.forward(p, b)
        L.backward(p, b)
        torch.cuda.synchronize()
        assert torch.equal(b.y.cpu(), ys[i]), f"y of step {i}"
        assert torch.equal(b.dx.cpu(), dxs[i]), f"dx of step {i}"
    assert torch.equal(b.dw_router, dwr_pipe)


STATS_SHAPES = [(1000, 16, 4, False), (4096, 128, 4, True), (300, 320, 2, False), (1, 8, 2, False),
                (777, 1024, 8, True)]


@pytest.mark.parametrize("T,E,k,dead", STATS_SHAPES, ids=lambda v: str(v))
def test_route_stats_parity(T, E, k, dead):
    """Routing load statistics vs the oracle on the GPU's own logits and counts.
    fp32 sums over at most ~100 partials per expert: 2e-5 relative."""
    rng = np.random.default_rng(T + E)
    logits = (rng.standard_normal((T, E)) * 2.0).astype(np.float32)
    if dead:
        logits[:, :3] -= 1e4  # three experts never selected
        logits[:, 5] += 3.0   # one busy expert
    b = L.Buffers(T, 64, E, k, 64, N.MOE_BF16)
    b.logits.copy_(torch.from_numpy(logits))
    N.moe_route(None, None, None, N.MOE_BF16, T, 64, E, k, b.logits, N.MOE_ROUTE_LOGITS_IN, b.topk_idx,
                b.gates, b.counts, b.offsets, b.dest_row, b.src_row, b.workspace)
    pm, st = L.route_stats(b)
    torch.cuda.synchronize()
    assert N.moe_get_device_error() == 0
    counts = b.counts.cpu().numpy()
    ref_pm, ref_st = oracle.route_stats(logits.astype(np.float64), counts, k)
    np.testing.assert_allclose(pm.cpu().numpy(), ref_pm, rtol=2e-5, atol=1e-9)
    got = st.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got[[0, 1, 3]], ref_st[[0, 1, 3]], rtol=2e-5, atol=1e-6)
    assert got[2] == ref_st[2]
    if dead:
        assert got[2] >= 3
    pm2, st2 = L.route_stats(b)
    assert torch.equal(pm, pm2) and torch.equal(st, st2)
