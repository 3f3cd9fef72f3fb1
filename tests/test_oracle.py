"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks the oracle against something independent of its code:
brute force, a library routine on a special case that reduces to it, central
finite differences, or the OCP E4M3/E8M0 specification tables. A plausible
slip anywhere in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong tie-break) fails at least one of these.
"""
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from mixture_experts_layer_prefix_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _silu(z):
    return z * scipy.special.expit(z)


def _dense_swiglu(x, wg, wu, wd):
    x = x.astype(np.float64)
    return (_silu(x @ wg) * (x @ wu)) @ wd


def _rand(rng, *shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (5, 5), (128, 4), (7, 1)])
def test_topk_matches_full_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    T = 300
    # coarse grid -> many exact ties, to pin the tie-break and the slot order
    l = np.round(rng.standard_normal((T, E)) * 4) / 4
    idx = oracle.topk(l, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -l[t]))  # by logit desc, then index asc
        assert list(idx[t]) == list(order[:k])
        assert len(set(idx[t])) == k


def test_gates_against_softmax_then_renormalise():
    rng = np.random.default_rng(1)
    T, E, k = 200, 16, 4
    l = rng.standard_normal((T, E)) * 3
    idx = oracle.topk(l, k)
    g = oracle.gates(l, idx)
    p = scipy.special.softmax(l, axis=1)
    ps = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(g, ps / ps.sum(1, keepdims=True), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(g.sum(1), 1.0, atol=1e-12)
    # descending gates follow descending logits
    assert np.all(np.diff(g, axis=1) <= 1e-15)


def test_gates_k_equals_E_is_softmax_and_k1_is_one():
    rng = np.random.default_rng(2)
    l = rng.standard_normal((50, 6)) * 2
    idx = oracle.topk(l, 6)
    g = oracle.gates(l, idx)
    p = scipy.special.softmax(l, axis=1)
    np.testing.assert_allclose(g, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=1e-13)
    g1 = oracle.gates(l, oracle.topk(l, 1))
    assert np.all(g1 == 1.0)


@pytest.mark.parametrize("E,k,T", [(8, 2, 512), (128, 4, 1000), (3, 3, 7), (16, 1, 1)])
def test_dispatch_matches_stable_sort(E, k, T):
    rng = np.random.default_rng(E + k + T)
    l = rng.standard_normal((T, E))
    if E > 4:
        l[:, :4] -= 100.0  # experts 0..3 never chosen: empty groups
    idx = oracle.topk(l, k)
    counts, offsets, dest, src = oracle.dispatch(idx, E)
    flat = idx.ravel().astype(np.int64)
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    order = np.argsort(flat, kind="stable")  # by expert, then by (token, slot)
    np.testing.assert_array_equal(src, order)
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    np.testing.assert_array_equal(dest.ravel(), inv)
    assert counts.sum() == T * k and offsets[-1] == T * k
    if E > 4:
        assert np.all(counts[:4] == 0)


# ------------------------------------------------------------ expert MLP
def test_E1_k1_is_dense_swiglu():
    rng = np.random.default_rng(3)
    T, d, f = 37, 24, 40
    x = _rand(rng, T, d)
    wg, wu = _rand(rng, 1, d, f, std=d ** -0.5), _rand(rng, 1, d, f, std=d ** -0.5)
    wd = _rand(rng, 1, f, d, std=f ** -0.5)
    wr = _rand(rng, d, 1)
    dy = _rand(rng, T, d)
    out = oracle.layer(x, wr, wg, wu, wd, dy, k=1)
    np.testing.assert_allclose(out["y"], _dense_swiglu(x, wg[0], wu[0], wd[0]), rtol=1e-12, atol=1e-12)
    assert np.all(out["gates"] == 1.0)
    # with one expert the router gets no gradient
    assert np.all(out["dlogits"] == 0.0) and np.all(out["dw_r"] == 0.0)
    # dense SwiGLU backward, written with matrix products (torch autograd, fp64)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    W = [torch.tensor(w[0], dtype=torch.float64, requires_grad=True) for w in (wg, wu, wd)]
    y = (torch.nn.functional.silu(xt @ W[0]) * (xt @ W[1])) @ W[2]
    (y * torch.tensor(dy, dtype=torch.float64)).sum().backward()
    np.testing.assert_allclose(out["dx"], xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["dw_gate"][0], W[0].grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["dw_up"][0], W[1].grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["dw_down"][0], W[2].grad.numpy(), rtol=1e-11, atol=1e-12)


def test_identical_experts_give_dense_mlp():
    rng = np.random.default_rng(4)
    T, d, f, E, k = 29, 16, 24, 6, 3
    x = _rand(rng, T, d)
    wg1, wu1 = _rand(rng, d, f, std=0.25), _rand(rng, d, f, std=0.25)
    wd1 = _rand(rng, f, d, std=0.2)
    wg, wu, wd = (np.repeat(w[None], E, 0) for w in (wg1, wu1, wd1))
    wr = _rand(rng, d, E)
    dy = _rand(rng, T, d)
    out = oracle.layer(x, wr, wg, wu, wd, dy, k=k)
    np.testing.assert_allclose(out["y"], _dense_swiglu(x, wg1, wu1, wd1), rtol=1e-11, atol=1e-12)
    # y does not depend on the gates, so the router gets no gradient
    np.testing.assert_allclose(out["dlogits"], 0.0, atol=1e-12)


def test_token_permutation_equivariance():
    rng = np.random.default_rng(5)
    T, d, f, E, k = 40, 16, 16, 8, 2
    x = _rand(rng, T, d)
    wg, wu = _rand(rng, E, d, f, std=0.25), _rand(rng, E, d, f, std=0.25)
    wd = _rand(rng, E, f, d, std=0.25)
    wr = _rand(rng, d, E)
    dy = _rand(rng, T, d)
    perm = rng.permutation(T)
    a = oracle.layer(x, wr, wg, wu, wd, dy, k)
    b = oracle.layer(x[perm], wr, wg, wu, wd, dy[perm], k)
    np.testing.assert_allclose(b["y"], a["y"][perm], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["dx"], a["dx"][perm], rtol=1e-12, atol=1e-13)
    for key in ("dw_gate", "dw_up", "dw_down", "dw_r"):
        np.testing.assert_allclose(b[key], a[key], rtol=1e-10, atol=1e-12)


def _margin_ok(l, k, margin):
    s = np.sort(l, axis=1)[:, ::-1]
    return np.all(s[:, k - 1] - s[:, k] > margin)


def test_backward_against_finite_differences():
    """Central differences in fp64 of L = <dy, y> w.r.t. every input and weight,
    on inputs whose k-th / (k+1)-th logit gap is large enough that no step of
    size h can change the selected experts."""
    T, d, E, k, f = 4, 8, 4, 2, 8
    rng = np.random.default_rng(6)
    while True:
        x = rng.standard_normal((T, d))
        wr = rng.standard_normal((d, E)) * 0.7
        if _margin_ok(x @ wr, k, 1e-3):
            break
    wg = rng.standard_normal((E, d, f)) * 0.4
    wu = rng.standard_normal((E, d, f)) * 0.4
    wd = rng.standard_normal((E, f, d)) * 0.4
    dy = rng.standard_normal((T, d))

    # the oracle takes float32 storage; run FD on the very same fp32 values
    x, wr, wg, wu, wd, dy = (a.astype(np.float32).astype(np.float64) for a in (x, wr, wg, wu, wd, dy))
    base = oracle.layer(x, wr, wg, wu, wd, dy, k)

    def loss(xx, wrr, wgg, wuu, wdd):
        # perturbations are applied in fp64 and passed as logits / weights below
        l = xx @ wrr
        r = oracle.route(l, k, E)
        fw = _forward64(xx, wgg, wuu, wdd, r["topk_idx"], r["gates"])
        return float((dy * fw).sum())

    h = 1e-6
    for name, arr, grad in (("x", x, base["dx"]), ("w_r", wr, base["dw_r"]),
                            ("w_gate", wg, base["dw_gate"]), ("w_up", wu, base["dw_up"]),
                            ("w_down", wd, base["dw_down"])):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            args = dict(x=x, w_r=wr, w_gate=wg, w_up=wu, w_down=wd)
            p = arr.copy(); p[i] += h
            m = arr.copy(); m[i] -= h
            args[name] = p
            lp = loss(args["x"], args["w_r"], args["w_gate"], args["w_up"], args["w_down"])
            args[name] = m
            lm = loss(args["x"], args["w_r"], args["w_gate"], args["w_up"], args["w_down"])
            num[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7, err_msg=name)

    # dlogits against finite differences on the logits themselves
    l0 = x @ wr
    num = np.zeros_like(l0)
    for t in range(T):
        for e in range(E):
            lp = l0.copy(); lp[t, e] += h
            lm = l0.copy(); lm[t, e] -= h
            fp = oracle.layer(x, wr, wg, wu, wd, dy, k, logits=lp)["y"]
            fm = oracle.layer(x, wr, wg, wu, wd, dy, k, logits=lm)["y"]
            num[t, e] = ((dy * fp).sum() - (dy * fm).sum()) / (2 * h)
    np.testing.assert_allclose(base["dlogits"], num, rtol=1e-6, atol=1e-8)
    # unselected experts get exactly zero
    sel = np.zeros((T, E), bool)
    np.put_along_axis(sel, base["topk_idx"].astype(np.int64), True, 1)
    assert np.all(base["dlogits"][~sel] == 0.0)


def _forward64(x, wg, wu, wd, idx, g):
    """Gate-weighted SwiGLU experts in fp64 numpy (used only by the FD pin, so
    that perturbations of size 1e-6 are not lost to float32 storage)."""
    T, d = x.shape
    y = np.zeros((T, d))
    for t in range(T):
        for j in range(idx.shape[1]):
            e = idx[t, j]
            y[t] += g[t, j] * _dense_swiglu(x[t:t + 1], wg[e], wu[e], wd[e])[0]
    return y


def test_forward_against_numpy_per_expert():
    """Forward y and the per-pair values against per-expert numpy matrix products."""
    s = synth.shape("tiny_fp32", T=64)
    inp = synth.Inputs(s, seed=3)
    x, wr, wg, wu, wd, dy = inp.x(), inp.w_r(), inp.w_gate(), inp.w_up(), inp.w_down(), inp.dy()
    out = oracle.layer(x, wr, wg, wu, wd, dy, s.k)
    xd = x.astype(np.float64)
    np.testing.assert_allclose(out["logits"], xd @ wr.astype(np.float64), rtol=1e-12, atol=1e-12)
    idx, g = out["topk_idx"], out["gates"]
    y = np.zeros((s.T, s.d))
    for t in range(s.T):
        for j in range(s.k):
            e = idx[t, j]
            hg = xd[t] @ wg[e].astype(np.float64)
            np.testing.assert_allclose(out["hg"][t * s.k + j], hg, rtol=1e-12, atol=1e-12)
            y[t] += g[t, j] * _dense_swiglu(xd[t:t + 1], wg[e].astype(np.float64),
                                            wu[e].astype(np.float64), wd[e].astype(np.float64))[0]
    np.testing.assert_allclose(out["y"], y, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------------ MXFP8
def test_e4m3_decode_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2  # 0x7F and 0xFF
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_e4m3_golden_spec_values():
    path = os.path.join(HERE, "golden", "e4m3_spec_values.txt")
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, val = line.split()
        code = int(code, 16)
        if val == "nan":
            assert np.isnan(oracle.e4m3_decode(code))
        else:
            v = float.fromhex(val) if "p" in val else float(val)
            assert oracle.e4m3_decode(code) == v, hex(code)
            if code not in (0x80,):
                assert oracle.e4m3_encode(v) == code, hex(code)
        n += 1
    assert n >= 10


def test_e4m3_encode_matches_torch_rounding():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(20000) * 0.01,
                        rng.uniform(-500, 500, 5000), np.array([0.0, 448.0, -448.0, 464.0, 1e-9])])
    # every representable value and every midpoint between neighbours (ties)
    tab = oracle.e4m3_table()
    pos = np.unique(tab[np.isfinite(tab) & (tab >= 0)])
    v = np.concatenate([v, pos, -pos, (pos[1:] + pos[:-1]) / 2, -(pos[1:] + pos[:-1]) / 2])
    ours = np.array([oracle.e4m3_encode(a) for a in v], np.uint8)
    ref = torch.tensor(np.clip(v, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_e8m0_exponent_is_smallest_unsaturated_power():
    rng = np.random.default_rng(8)
    am = np.concatenate([np.exp(rng.uniform(-60, 60, 5000)), [448.0, 449.0, 1.0, 2 ** -100, 896.0, 897.0]])
    for a in am:
        s = oracle.e8m0_exponent(a)
        assert a / 2.0 ** s <= 448.0
        assert a / 2.0 ** (s - 1) > 448.0
    assert oracle.e8m0_exponent(0.0) == -127
    assert oracle.e8m0_exponent(448.0) == 0 and oracle.e8m0_exponent(449.0) == 1
    assert oracle.e8m0_exponent(1e300) == 127


def test_mxfp8_quantize_rows_against_torch_cast():
    rng = np.random.default_rng(9)
    v = synth.round_bf16((rng.standard_normal((40, 256)) * np.exp(rng.uniform(-8, 8, (40, 1)))).astype(np.float32))
    v[3, 32:64] = 0.0  # an all-zero block
    q, s = oracle.mxfp8_quantize_rows(v)
    assert s[3, 1] == 0 and np.all(q[3, 32:64] == 0)
    blocks = v.reshape(40, 8, 32).astype(np.float64)
    scaled = blocks * np.ldexp(1.0, 127 - s.astype(np.int32))[..., None]
    assert np.abs(scaled).max() <= 448.0
    ref = torch.tensor(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(40, 256)
    np.testing.assert_array_equal(q, ref)
    # error bound: half a step of the E4M3 grid at each element's magnitude
    deq = oracle.mxfp8_dequantize_rows(q, s)
    sc = np.repeat(np.ldexp(1.0, s.astype(np.int32) - 127), 32, axis=1)
    err = np.abs(deq - v) / sc
    mag = np.abs(v) / sc
    bound = np.where(mag >= 2 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(mag, 2 ** -6))) - 4), 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-12))


def test_mxfp8_exact_values_round_trip():
    tab = oracle.e4m3_table()
    vals = tab[np.isfinite(tab)]
    rng = np.random.default_rng(10)
    v = rng.choice(vals, size=(16, 64)).astype(np.float32)
    v[:, ::32] = 448.0  # block max pinned so that the scale exponent is 0
    q, s = oracle.mxfp8_quantize_rows(v)
    assert np.all(s == 127)
    np.testing.assert_array_equal(oracle.mxfp8_dequantize_rows(q, s), v.astype(np.float64))


def test_mxfp8_segmented_columns_equal_rows_of_padded_transpose():
    rng = np.random.default_rng(11)
    seg = np.array([0, 5, 5, 70, 100], np.int32)  # includes an empty segment and ragged tails
    v = synth.round_bf16(rng.standard_normal((100, 64)).astype(np.float32))
    q, s = oracle.mxfp8_quantize_cols_segmented(v, seg)
    brow = 0
    for g in range(len(seg) - 1):
        r0, r1 = seg[g], seg[g + 1]
        n = r1 - r0
        if n == 0:
            continue
        nb = (n + 31) // 32
        pad = np.zeros((nb * 32, 64), np.float32)
        pad[:n] = v[r0:r1]
        qt, st = oracle.mxfp8_quantize_rows(np.ascontiguousarray(pad.T))
        np.testing.assert_array_equal(q[r0:r1], qt.T[:n])
        np.testing.assert_array_equal(s[brow:brow + nb], st.T)
        brow += nb
    assert brow == s.shape[0]


# --------------------------------------------------------- MXFP8 layer oracle
def test_mxfp8_layer_without_quantisation_is_the_c_oracle():
    """The MXFP8 layer oracle with its fake-quantisations switched off must equal
    the token-by-token C oracle on every output (per-pair values compared in
    dispatch order)."""
    from oracle import mxfp8_layer
    rng = np.random.default_rng(12)
    T, d, E, k, f = 50, 64, 6, 2, 32
    x = _rand(rng, T, d)
    wr = _rand(rng, d, E)
    wg, wu = _rand(rng, E, d, f, std=0.2), _rand(rng, E, d, f, std=0.2)
    wd = _rand(rng, E, f, d, std=0.2)
    dy = _rand(rng, T, d)
    logits = x.astype(np.float64) @ wr.astype(np.float64)
    logits[:, 0] -= 50.0  # expert 0 empty
    ref = oracle.layer(x, wr, wg, wu, wd, dy, k, logits=logits)
    got = mxfp8_layer.layer(x, wr, wg, wu, wd, dy, k, logits, quant=False, store_bf16=False)
    dest = ref["dest_row"].ravel()
    np.testing.assert_allclose(got["hg"][dest], ref["hg"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(got["ye"][dest], ref["ye"], rtol=1e-11, atol=1e-12)
    for key in ("y", "dgates", "dlogits", "dx", "dw_gate", "dw_up", "dw_down", "dw_r"):
        np.testing.assert_allclose(got[key], ref[key], rtol=1e-10, atol=1e-11, err_msg=key)


def test_mxfp8_fakequant_f64_matches_f32_quantiser():
    rng = np.random.default_rng(13)
    v = synth.round_bf16((rng.standard_normal((64, 128)) * 3).astype(np.float32))
    q, s = oracle.mxfp8_quantize_rows(v)
    np.testing.assert_array_equal(oracle.mxfp8_fakequant_rows(v.astype(np.float64)),
                                  oracle.mxfp8_dequantize_rows(q, s))
    seg = np.array([0, 10, 10, 64], np.int32)
    q, s = oracle.mxfp8_quantize_cols_segmented(v, seg)
    np.testing.assert_array_equal(oracle.mxfp8_fakequant_cols_segmented(v.astype(np.float64), seg),
                                  oracle.mxfp8_dequantize_cols_segmented(q, s, seg))


def test_mxfp8_layer_close_to_unquantised():
    """Quantisation error of the whole MXFP8 layer stays at the few-percent level
    E4M3 implies (3 mantissa bits: relative step 2^-3, error <= 2^-4 per element)."""
    from oracle import mxfp8_layer
    rng = np.random.default_rng(14)
    T, d, E, k, f = 64, 64, 4, 2, 64
    x = synth.round_bf16(rng.standard_normal((T, d)).astype(np.float32))
    wr = _rand(rng, d, E, std=0.2)
    wg, wu = _rand(rng, E, d, f, std=d ** -0.5), _rand(rng, E, d, f, std=d ** -0.5)
    wd = _rand(rng, E, f, d, std=f ** -0.5)
    dy = _rand(rng, T, d)
    logits = x.astype(np.float64) @ wr.astype(np.float64)
    a = mxfp8_layer.layer(x, wr, wg, wu, wd, dy, k, logits, quant=True, store_bf16=False)
    b = mxfp8_layer.layer(x, wr, wg, wu, wd, dy, k, logits, quant=False, store_bf16=False)
    for key in ("y", "dx", "dw_gate", "dw_down"):
        err = np.abs(a[key] - b[key]).max() / np.abs(b[key]).max()
        assert 1e-4 < err < 0.1, (key, err)


def test_mxfp8_oracle_bf16_rounding_matches_library():
    from oracle import mxfp8_layer
    rng = np.random.default_rng(15)
    v = rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))
    ref = torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(mxfp8_layer.round_bf16(v), ref)


# ---------------------------------------------------------------- routing load statistics
def test_route_stats_uniform_and_balanced():
    T, E, k = 96, 8, 2
    pm, st = oracle.route_stats(np.zeros((T, E)), np.full(E, T * k // E, np.int32), k)
    np.testing.assert_allclose(pm, np.full(E, 1.0 / E), rtol=0, atol=1e-15)
    np.testing.assert_allclose(st, [1.0, 1.0, 0.0, 0.0], rtol=0, atol=1e-15)


def test_route_stats_all_tokens_on_one_expert_closed_forms():
    T, E, k = 50, 6, 1
    logits = np.zeros((T, E))
    logits[:, 2] = 3.0
    counts = np.zeros(E, np.int32)
    counts[2] = T
    pm, st = oracle.route_stats(logits, counts, k)
    p2 = np.exp(3.0) / (np.exp(3.0) + (E - 1))
    assert abs(pm[2] - p2) < 1e-15
    assert abs(st[0] - E * p2) < 1e-13           # E * f_2 * P_2 with f_2 = 1
    assert st[1] == E                             # T / (T / E)
    assert st[2] == E - 1
    assert abs(st[3] - np.sqrt(E - 1)) < 1e-12    # std / mean of (T, 0, ..., 0)


def test_route_stats_matches_library_softmax_and_is_label_invariant():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(4)
    T, E, k = 200, 12, 3
    logits = rng.standard_normal((T, E)) * 2.0
    counts = rng.integers(0, 90, E).astype(np.int32)
    pm, st = oracle.route_stats(logits, counts, k)
    np.testing.assert_allclose(pm, special.softmax(logits, axis=1).mean(axis=0), rtol=1e-13, atol=0)
    assert abs(pm.sum() - 1.0) < 1e-13
    perm = rng.permutation(E)
    pm2, st2 = oracle.route_stats(logits[:, perm], counts[perm], k)
    np.testing.assert_allclose(pm2, pm[perm], rtol=1e-13, atol=0)
    np.testing.assert_allclose(st2, st, rtol=1e-12, atol=0)


# ------------------------------------- MXFP8 layer oracle: operand blocking of each GEMM
# tests/mx_exact_inputs.py builds, per expert GEMM, inputs whose operands are
# exactly representable under the blocking the oracle states for that GEMM and
# lose a whole binade band under the transposed blocking. Three pins per GEMM:
#   1. the oracle's quantised layer gives that GEMM's output bit for bit equal
#      to its unquantised layer (its blocking keeps every value);
#   2. the same GEMM with one operand blocked along the other axis (computed
#      here from the oracle's own quantisers) loses a band: some output row or
#      column changes by more than half its size -- so the oracle cannot be
#      using that blocking;
#   3. one input element given a 5-bit mantissa (17 * 2^p, not in E4M3) changes
#      that GEMM's output -- so the operand is quantised at all.
import mx_exact_inputs as MXI  # noqa: E402


def _mx_run(c, quant):
    from oracle import mxfp8_layer
    return mxfp8_layer.layer(c["x"], c["w_r"], c["w_gate"], c["w_up"], c["w_down"], c["dy"], c["k"], c["logits"],
                             quant=quant, store_bf16=False)


def _slice_err(got, ref, how):
    """Largest per-row ("row") or per-column ("col") error, each slice normalised by
    its own largest reference magnitude (slices that are zero in both are skipped)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    ax = -1 if how == "row" else -2
    num = np.abs(got - ref).max(axis=ax)
    den = np.abs(ref).max(axis=ax)
    keep = (den > 0) | (num > 0)
    return float((num[keep] / np.where(den[keep] > 0, den[keep], 1e-300)).max()) if keep.any() else 0.0


def _blocked(v, axis, offsets=None):
    """The oracle's MXFP8 fake-quantisation of v: 'k' = blocks of 32 along the last
    axis; 'seg' = blocks of 32 rows from each expert segment's start; 'w' = blocks
    of 32 rows of a single weight matrix."""
    if axis == "k":
        return oracle.mxfp8_fakequant_rows(v)
    if axis == "seg":
        return oracle.mxfp8_fakequant_cols_segmented(v, offsets)
    return oracle.mxfp8_fakequant_cols_segmented(v, np.array([0, v.shape[0]], np.int32))


def _gemm_out(name, r, c, a_axis, b_axis):
    """The targeted GEMM recomputed from the unquantised run's operands, operand A
    blocked along a_axis and B along b_axis (None: not quantised)."""
    q = lambda v, ax, offs=None: v if ax is None else _blocked(v, ax, offs)  # noqa: E731
    offs = r["offsets"]
    E = c["w_gate"].shape[0]
    f = c["w_gate"].shape[2]
    segs = [(e, int(offs[e]), int(offs[e + 1])) for e in range(E) if offs[e + 1] > offs[e]]
    xp = np.asarray(c["x"], np.float64)[r["src_row"] // c["k"]]
    if name == "gemm1":
        A, out = q(xp, a_axis, offs), np.zeros_like(r["hg"])
        for e, r0, r1 in segs:
            out[r0:r1] = A[r0:r1] @ q(c["w_gate"][e], b_axis)
        return out
    if name == "gemm2":
        A, out = q(r["a"], a_axis, offs), np.zeros_like(r["ye"])
        for e, r0, r1 in segs:
            out[r0:r1] = A[r0:r1] @ q(c["w_down"][e], b_axis)
        return out
    if name.startswith("dgrad2"):  # da = dye . w_down^T (da is what dh is made of)
        A, out = q(r["dye"], a_axis, offs), np.zeros((r["dye"].shape[0], f))
        for e, r0, r1 in segs:
            out[r0:r1] = A[r0:r1] @ q(c["w_down"][e], b_axis).T
        return out
    if name == "wgrad2":
        A, B = q(r["a"], a_axis, offs), q(r["dye"], b_axis, offs)
        out = np.zeros_like(r["dw_down"])
        for e, r0, r1 in segs:
            out[e] = A[r0:r1].T @ B[r0:r1]
        return out
    if name == "dgrad1":
        A, out = q(r["dh"], a_axis, offs), np.zeros_like(r["dx_perm"])
        for e, r0, r1 in segs:
            out[r0:r1] = A[r0:r1, :f] @ q(c["w_gate"][e], b_axis).T + A[r0:r1, f:] @ q(c["w_up"][e], b_axis).T
        return out
    if name == "wgrad1":
        A, B = q(xp, a_axis, offs), q(r["dh"], b_axis, offs)
        out = np.zeros_like(r["dw_gate"])
        for e, r0, r1 in segs:
            out[e] = A[r0:r1].T @ B[r0:r1, :f]
        return out
    raise KeyError(name)


# per case: the stated blocking of (A, B), and the transposed one of each
_MX_AXES = {"gemm1": ("k", "w"), "gemm2": ("k", "w"), "dgrad2_w": ("k", "k"), "dgrad2_dy": ("k", "k"),
            "wgrad2": ("seg", "seg"), "dgrad1": ("k", "k"), "wgrad1": ("seg", "seg")}
_MX_WRONG = {"k": "seg", "seg": "k", "w": "k"}
_MX_WRONG_B = {"gemm1": "k", "gemm2": "k", "dgrad2_w": "w", "dgrad2_dy": "w", "wgrad2": "k", "dgrad1": "w",
               "wgrad1": "k"}
# which operands each case discriminates (dgrad2 needs one case per operand)
_MX_OPS = {"dgrad2_w": ("B",), "dgrad2_dy": ("A",)}


@pytest.mark.parametrize("name", list(MXI.TARGETS))
def test_mxfp8_oracle_blocking_is_exact_as_stated_and_not_transposed(name):
    c = MXI.case(name)
    rq, rp = _mx_run(c, True), _mx_run(c, False)
    gemm, ops = MXI.TARGETS[name]
    np.testing.assert_array_equal(rq["offsets"], [0, 67, 134, 200, 200])  # ragged segments, one empty
    # 1. the oracle's quantised GEMM output is the unquantised one, bit for bit
    for _, key, _ in ops:
        np.testing.assert_array_equal(rq[key], rp[key], err_msg=f"{gemm}: {key}")
    # the stated blocking recomputed here is exact too; with no quantisation at all it is the same product
    a_ax, b_ax = _MX_AXES[name]
    exact = _gemm_out(name, rp, c, None, None)
    np.testing.assert_array_equal(_gemm_out(name, rp, c, a_ax, b_ax), exact)
    # 2. each operand blocked along the other axis loses a band
    which = _MX_OPS.get(name, ("A", "B"))
    for (desc, key, how), op in zip(ops, which):
        if op == "A":
            alt = _gemm_out(name, rp, c, _MX_WRONG[a_ax], b_ax)
        else:
            alt = _gemm_out(name, rp, c, a_ax, _MX_WRONG_B[name])
        assert _slice_err(alt, exact, how) > 0.5, f"{gemm}: {desc} transposed is not detected"


# per case: an input element given a 5-bit mantissa, and the output that must change
_MX_PERTURB = {"gemm1": [("x", (4, 9), "hg"), ("w_gate", (0, 3, 5), "hg")],
               "gemm2": [("w_down", (1, 6, 2), "ye")],
               "dgrad2_w": [("w_down", (0, 6, 0), "dh")],  # token 0: expert 0, dy at column 0
               "dgrad2_dy": [("dy", (10, 5), "dh")],
               "wgrad2": [("dy", (7, 4), "dw_down")],
               "dgrad1": [("w_gate", (2, 8, 6), "dx_perm")],
               "wgrad1": [("x", (3, 2 * ((7 * 3) % 64) + 1), "dw_gate")]}


@pytest.mark.parametrize("name", list(MXI.TARGETS))
def test_mxfp8_oracle_quantises_each_input_operand(name):
    for key, idx, out in _MX_PERTURB[name]:
        c = MXI.case(name)
        v = c[key][idx]
        assert v != 0.0
        p = np.floor(np.log2(abs(v)))
        c[key] = c[key].copy()
        c[key][idx] = np.sign(v) * 17.0 * 2.0 ** (p - 4)  # 5 significant bits, same binade as before
        rq, rp = _mx_run(c, True), _mx_run(c, False)
        assert np.any(rq[out] != rp[out]), (name, key, out)
