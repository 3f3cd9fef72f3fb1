"""Parity at the workloads' full sizes, in the launch configuration bench.py
times, on outputs the oracle computes one by one.

For each workload the whole layer runs forward+backward on the GPU; then
  - routing metadata is compared bit-exactly over all T tokens, with the
    oracle routing on the GPU's own fp32 logits;
  - router logits of sampled tokens against the oracle's fp64 router GEMM;
  - y, dx, dgates, dlogits of sampled tokens against the oracle restricted to
    the experts those tokens use (exact: other experts do not touch them);
  - weight gradients of sampled experts, from an oracle call that routes
    exactly that expert's tokens to it with their gates (dW_e depends on
    nothing else).
The router weight gradient is a per-expert sum of dlogits-weighted rows; its
kernel is compared element by element on the small shapes of
test_gpu_parity.py, and here through the sampled dlogits it reduces.
"""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_prefix_gb300 import _native as N
from mixture_experts_layer_prefix_gb300 import build as B
from mixture_experts_layer_prefix_gb300 import layer as L
from mixture_experts_layer_prefix_gb300 import synth

from helpers import BF16_TOL, maxnorm_err, np_of

pytestmark = pytest.mark.gpu

WORKLOADS = {  # name -> (token sample size, experts sampled for dW, max rows of a sampled expert)
    "e8_top4": (64, 1, 1 << 30),
    "e128_top4": (64, 3, 1 << 30),
    "e128_top4_skew": (64, 3, 1 << 30),
    "e128_top4_bf16_twin": (32, 2, 1 << 30),
    "stress_e256_top8": (8, 2, 1024),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    N.load()


def _token_sample_check(inp, b, gl, ref_route, tokens):
    s = inp.s
    idx = ref_route["topk_idx"][tokens]
    used = np.unique(idx)
    local = np.searchsorted(used, idx).astype(np.int32)
    x, dy = inp.x()[tokens], inp.dy()[tokens]
    w = inp.for_experts(used)
    wr = inp.w_r()[:, used]
    g = ref_route["gates"][tokens]
    fw = oracle.forward(x, w["w_gate"], w["w_up"], w["w_down"], local, g)
    bw = oracle.backward(x, wr, w["w_gate"], w["w_up"], w["w_down"], dy, local, g, fw)
    dl_full = np.zeros((len(tokens), s.E))
    dl_full[:, used] = bw["dlogits"]
    errs = {
        "y": maxnorm_err(np_of(b.y)[tokens], fw["y"]),
        "dx": maxnorm_err(np_of(b.dx)[tokens], bw["dx"]),
        "dgates": maxnorm_err(np_of(b.dgates)[tokens], bw["dgates"]),
        "dlogits": maxnorm_err(np_of(b.dlogits)[tokens], dl_full),
    }
    return errs


def _expert_dw_check(inp, b, ref_route, e):
    """dW of expert e: oracle calls that route exactly e's tokens to it with
    their gates; the rows are split in chunks (run concurrently, summed in
    chunk order) so that large experts stay quick."""
    s = inp.s
    idx, g = ref_route["topk_idx"], ref_route["gates"]
    tok, slot = np.nonzero(idx == e)
    w = inp.for_experts([e])
    ge_all = g[tok, slot][:, None]
    chunks = np.array_split(np.arange(len(tok)), max(1, min(16, len(tok) // 128)))

    def run(ch):
        t = tok[ch]
        zeros = np.zeros((len(ch), 1), np.int32)
        ge = ge_all[ch]
        x, dy = inp.x()[t], inp.dy()[t]
        fw = oracle.forward(x, w["w_gate"], w["w_up"], w["w_down"], zeros, ge, nthreads=1)
        bw = oracle.backward(x, np.zeros((s.d, 1), np.float32), w["w_gate"], w["w_up"], w["w_down"], dy,
                             zeros, ge, fw, nthreads=1)
        return bw["dw_gate"][0], bw["dw_up"][0], bw["dw_down"][0]

    with cf.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        parts = list(ex.map(run, chunks))
    dwg = sum(p_[0] for p_ in parts)
    dwu = sum(p_[1] for p_ in parts)
    dwd = sum(p_[2] for p_ in parts)
    return {
        f"dw_gate[{e}]": maxnorm_err(np_of(b.dw_gate[e]), dwg),
        f"dw_up[{e}]": maxnorm_err(np_of(b.dw_up[e]), dwu),
        f"dw_down[{e}]": maxnorm_err(np_of(b.dw_down[e]), dwd),
    }


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_fullsize_sampled_parity(name):
    s = synth.CONFIGS[name]
    n_tok, n_exp, max_rows = WORKLOADS[name]
    inp = synth.Inputs(s, seed=0)
    p = L.params_from_inputs(inp, N.MOE_BF16)
    b = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_BF16)
    L.forward(p, b)
    L.backward(p, b)
    torch.cuda.synchronize()
    assert N.moe_get_device_error() == 0

    gl = b.logits.cpu().numpy()
    ref_route = oracle.route(gl.astype(np.float64), s.k, s.E)
    for key in ("topk_idx", "counts", "offsets", "dest_row", "src_row"):
        np.testing.assert_array_equal(getattr(b, key).cpu().numpy(), ref_route[key], err_msg=key)
    np.testing.assert_allclose(b.gates.cpu().numpy(), ref_route["gates"], rtol=0, atol=2e-6)
    assert int(b.offsets[-1]) == s.T * s.k

    rng = np.random.default_rng(123)
    tokens = np.sort(rng.choice(s.T, size=n_tok, replace=False))
    ref_l = oracle.router_logits(inp.x()[tokens], inp.w_r(), inp.bias())
    assert maxnorm_err(gl[tokens], ref_l) < 1e-5

    errs = _token_sample_check(inp, b, gl, ref_route, tokens)
    counts = ref_route["counts"]
    cand = np.flatnonzero((counts > 0) & (counts <= max_rows))
    picks = [int(cand[np.argmin(counts[cand])]), int(cand[np.argmax(counts[cand])])]
    picks += [int(e) for e in rng.choice(cand, size=max(0, n_exp - 2), replace=False)]
    for e in sorted(set(picks))[:max(n_exp, 1)]:
        errs.update(_expert_dw_check(inp, b, ref_route, e))
    empty = np.flatnonzero(counts == 0)
    for e in empty[:2]:
        assert float(b.dw_gate[int(e)].float().abs().max()) == 0.0
    bad = {k: v for k, v in errs.items() if not v <= BF16_TOL}
    assert not bad, f"{name}: {bad} (all: {errs})"


@pytest.mark.parametrize("pairs", [0, 1], ids=["single_cta", "cta_pairs"])
def test_fullsize_mxfp8_sampled_parity(pairs):
    """The MXFP8 workload (T=32768, E=128, k=4) at full size, run as bench.py
    runs it (weights prepared, rows quantised where produced; the weight
    gradients on single CTAs or, with pairs, as bench.py --cta-pairs): routing exact;
    y, dx, dgates, dlogits of sampled tokens and the weight gradients of
    sampled experts against the MXFP8 oracle on the same dequantised operands.
    Every quantisation the oracle applies is local to what is sampled: token
    rows along d, f and 2f; weights per matrix; the weight-gradient operands
    along one expert's rows (its tokens in token order, as in the layer)."""
    from oracle import mxfp8_layer

    s = synth.CONFIGS["e128_top4_mxfp8"]
    inp = synth.Inputs(s, seed=0)
    p = L.params_from_inputs(inp, N.MOE_MXFP8)
    b = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_MXFP8)
    N.moe_use_cta_pairs(pairs)
    try:
        L.forward(p, b)
        L.backward(p, b)
        torch.cuda.synchronize()
    finally:
        N.moe_use_cta_pairs(0)
    assert N.moe_get_device_error() == 0

    gl = b.logits.cpu().numpy().astype(np.float64)
    ref_route = oracle.route(gl, s.k, s.E)
    for key in ("topk_idx", "counts", "offsets", "dest_row", "src_row"):
        np.testing.assert_array_equal(getattr(b, key).cpu().numpy(), ref_route[key], err_msg=key)

    tol = 6e-2
    rng = np.random.default_rng(321)
    tokens = np.sort(rng.choice(s.T, size=8, replace=False))
    used = np.unique(ref_route["topk_idx"][tokens])
    w = inp.for_experts(used)
    ref = mxfp8_layer.layer(inp.x()[tokens], inp.w_r()[:, used], w["w_gate"], w["w_up"], w["w_down"],
                            inp.dy()[tokens], s.k, gl[tokens][:, used])
    dl_full = np.zeros((len(tokens), s.E))
    dl_full[:, used] = ref["dlogits"]
    errs = {
        "y": maxnorm_err(np_of(b.y)[tokens], ref["y"]),
        "dx": maxnorm_err(np_of(b.dx)[tokens], ref["dx"]),
        "dgates": maxnorm_err(np_of(b.dgates)[tokens], ref["dgates"]),
        "dlogits": maxnorm_err(np_of(b.dlogits)[tokens], dl_full),
    }
    counts = ref_route["counts"]
    cand = np.flatnonzero(counts > 0)
    for e in (int(cand[np.argmin(counts[cand])]), int(cand[np.argmax(counts[cand])])):
        tok, slot = np.nonzero(ref_route["topk_idx"] == e)
        ge = ref_route["gates"][tok, slot][:, None]
        we = inp.for_experts([e])
        # one expert, k = 1: gate 1, so dy is pre-scaled by the layer's gates
        r1 = mxfp8_layer.layer(inp.x()[tok], np.zeros((s.d, 1)), we["w_gate"], we["w_up"], we["w_down"],
                               ge * inp.dy()[tok].astype(np.float64), 1, np.zeros((len(tok), 1)))
        errs[f"dw_gate[{e}]"] = maxnorm_err(np_of(b.dw_gate[e]), r1["dw_gate"][0])
        errs[f"dw_up[{e}]"] = maxnorm_err(np_of(b.dw_up[e]), r1["dw_up"][0])
        errs[f"dw_down[{e}]"] = maxnorm_err(np_of(b.dw_down[e]), r1["dw_down"][0])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{bad} (all: {errs})"


@pytest.mark.parametrize("name", ["e128_top4", "e128_top4_skew"])
def test_fullsize_cta_pair_weight_gradients(name):
    """The weight gradients on CTA pairs (moe_use_cta_pairs(1)) at the
    workload's full size, in the launch configuration bench.py --cta-pairs
    times: the smallest, the largest and one more sampled expert against the
    oracle, and exact zeros for experts without rows."""
    s = synth.CONFIGS[name]
    inp = synth.Inputs(s, seed=0)
    p = L.params_from_inputs(inp, N.MOE_BF16)
    b = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_BF16)
    N.moe_use_cta_pairs(1)
    try:
        L.forward(p, b)
        L.backward(p, b)
        torch.cuda.synchronize()
    finally:
        N.moe_use_cta_pairs(0)
    assert N.moe_get_device_error() == 0
    gl = b.logits.cpu().numpy()
    ref_route = oracle.route(gl.astype(np.float64), s.k, s.E)
    np.testing.assert_array_equal(b.offsets.cpu().numpy(), ref_route["offsets"])
    counts = ref_route["counts"]
    cand = np.flatnonzero(counts > 0)
    rng = np.random.default_rng(7)
    picks = {int(cand[np.argmin(counts[cand])]), int(cand[np.argmax(counts[cand])]), int(rng.choice(cand))}
    errs = {}
    for e in sorted(picks):
        errs.update(_expert_dw_check(inp, b, ref_route, e))
    for e in np.flatnonzero(counts == 0)[:2]:
        assert float(b.dw_gate[int(e)].float().abs().max()) == 0.0
        assert float(b.dw_down[int(e)].float().abs().max()) == 0.0
    bad = {k: v for k, v in errs.items() if not v <= BF16_TOL}
    assert not bad, f"{name}: {bad} (all: {errs})"
