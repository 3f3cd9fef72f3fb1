"""fp64 oracle of the MoE layer with MXFP8 expert GEMMs -- TEST INFRASTRUCTURE.

Same layer as the C oracle ("Introducing Olmo-core 3", section "Scaling and
optimizing MoE training": MXFP8 for the expert feed-forward), with every
operand of the six expert GEMMs replaced by its MXFP8 value along that GEMM's
K: dequantise(quantise(v)), E4M3 elements with one E8M0 scale per 32
elements (the C oracle's spec quantiser). Routing, gates, SwiGLU, the combine
and the router backward stay in fp64 on unquantised values. Operands:

  GEMM1  x rows along d;            w_gate, w_up along d (32-row blocks)
  GEMM2  a rows along f;            w_down along f
  dgrad2 dye rows along d;          w_down along d (its rows)
  wgrad2 a, dye along the expert's rows (blocks of 32 rows from the segment start)
  dgrad1 dh rows along 2f;          w_gate, w_up along f (their rows)
  wgrad1 x, dh along the expert's rows

Each GEMM is a per-expert matrix product over that expert's rows in dispatch
order. Activations are stored in bf16 between steps, as on the bf16 path
(store_bf16=True): h = (hg | hu), a, the expert outputs, dye, dh and dx_perm
are rounded to bf16 (nearest, ties to even) where they are stored, and later
steps read the stored values; the arithmetic itself stays fp64. With
quant=False and store_bf16=False every fake-quantisation and rounding is the
identity and the function must equal the C oracle (its pin).
"""
from __future__ import annotations

import numpy as np

from . import dispatch, gates as gates_fn, topk, mxfp8_fakequant_cols_segmented, mxfp8_fakequant_rows


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _dsilu(z):
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def round_bf16(v):
    """Round fp64 values to the nearest bfloat16 (8 significant bits, ties to even)."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)                 # v = m * 2^e, |m| in [0.5, 1)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def layer(x, w_r, w_gate, w_up, w_down, dy, k, logits, quant=True, store_bf16=True):
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    w_r = np.asarray(w_r, np.float64)
    wg, wu, wd = (np.asarray(w, np.float64) for w in (w_gate, w_up, w_down))
    T, d = x.shape
    E, _, f = wg.shape
    logits = np.asarray(logits, np.float64)
    idx = topk(logits, k)
    g = gates_fn(logits, idx)
    counts, offsets, dest, src = dispatch(idx, E)
    R = T * k
    tok = src // k          # token of each dispatched row
    gr = g.ravel()[src]     # gate of each dispatched row

    fq_rows = mxfp8_fakequant_rows if quant else (lambda v: np.asarray(v, np.float64))
    st = round_bf16 if store_bf16 else (lambda v: np.asarray(v, np.float64))

    def fq_seg(v):
        return mxfp8_fakequant_cols_segmented(v, offsets) if quant else np.asarray(v, np.float64)

    def fq_wcols(w):  # one expert's [K][N] weight, blocks of 32 rows
        if not quant:
            return w
        return mxfp8_fakequant_cols_segmented(w, np.array([0, w.shape[0]], np.int32))

    xp = x[tok]
    xq = fq_rows(xp)
    hg = np.zeros((R, f)); hu = np.zeros((R, f)); ye = np.zeros((R, d))
    segs = [(e, int(offsets[e]), int(offsets[e + 1])) for e in range(E) if offsets[e + 1] > offsets[e]]
    for e, r0, r1 in segs:
        hg[r0:r1] = xq[r0:r1] @ fq_wcols(wg[e])
        hu[r0:r1] = xq[r0:r1] @ fq_wcols(wu[e])
    a = st(_silu(hg) * hu)
    hg, hu = st(hg), st(hu)
    aq = fq_rows(a)
    for e, r0, r1 in segs:
        ye[r0:r1] = aq[r0:r1] @ fq_wcols(wd[e])
    ye = st(ye)
    y = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            y[t] += g[t, j] * ye[dest[t, j]]

    # backward
    dye = st(gr[:, None] * dy[tok])
    dgates = np.zeros((T, k))
    for t in range(T):
        for j in range(k):
            dgates[t, j] = dy[t] @ ye[dest[t, j]]
    dyq = fq_rows(dye)
    da = np.zeros((R, f))
    for e, r0, r1 in segs:
        da[r0:r1] = dyq[r0:r1] @ fq_rows(wd[e]).T
    dhg = da * hu * _dsilu(hg)
    dhu = da * _silu(hg)
    dh = st(np.concatenate([dhg, dhu], axis=1))
    dhq = fq_rows(dh)
    dx_perm = np.zeros((R, d))
    dw_gate = np.zeros_like(wg); dw_up = np.zeros_like(wu); dw_down = np.zeros_like(wd)
    a_s, dye_s, x_s, dh_s = fq_seg(a), fq_seg(dye), fq_seg(xp), fq_seg(dh)
    for e, r0, r1 in segs:
        dx_perm[r0:r1] = dhq[r0:r1, :f] @ fq_rows(wg[e]).T + dhq[r0:r1, f:] @ fq_rows(wu[e]).T
        dw_down[e] = a_s[r0:r1].T @ dye_s[r0:r1]
        dw_gate[e] = x_s[r0:r1].T @ dh_s[r0:r1, :f]
        dw_up[e] = x_s[r0:r1].T @ dh_s[r0:r1, f:]
    # router: softmax over the selected logits
    dx_perm = st(dx_perm)
    dlogits = np.zeros((T, E))
    for t in range(T):
        for i in range(k):
            dlogits[t, idx[t, i]] = sum(dgates[t, j] * g[t, j] * ((i == j) - g[t, i]) for j in range(k))
    dx = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            dx[t] += dx_perm[dest[t, j]]
    dx += dlogits @ w_r.T
    dw_r = x.T @ dlogits
    return dict(topk_idx=idx, gates=g, offsets=offsets, dest_row=dest, src_row=src, hg=hg, hu=hu, a=a, ye=ye,
                y=y, dye=dye, dgates=dgates, dh=dh, dx_perm=dx_perm, dlogits=dlogits, dx=dx, dw_gate=dw_gate,
                dw_up=dw_up, dw_down=dw_down, dw_r=dw_r)
