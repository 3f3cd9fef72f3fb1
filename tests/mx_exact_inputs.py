"""Layer inputs on which each MXFP8 expert GEMM is exact under the stated
operand blocking and inexact under the transposed one (test helper; it only
builds inputs and computes none of the layer).

The MXFP8 format keeps 4 significant bits (E4M3) under one power-of-two scale
per block of 32 elements. A value m * 2^P with an integer 1 <= m <= 15 is
therefore stored exactly when every element of its block lies in the same
binade band (their scale can then keep all of them in E4M3's normal range).
A block that mixes a 2^0 band with a 2^-20 band rounds the small band to zero.
So an operand whose band depends only on one index is exact when its blocks
run along the other index, and loses the small band when they run along the
first. Every case below gives the GEMM it targets such operands, and keeps the
GEMMs upstream of it exact as well:

  - x one-hot rows with a power-of-two value: the GEMM1 products are single
    products, so h_gate = m * 2^(6+...) >= 64 and h_up = +-2^(...) exactly;
  - h_gate >= 64 makes silu(h) = h and silu'(h) = 1 exactly in both fp64 and
    fp32 (exp(-64) vanishes against 1), so a = h_gate * h_up,
    dh_gate = da * h_up and dh_up = da * h_gate stay products of few bits;
  - logits with two equal maxima per token make both gates exactly 1/2;
  - expert E-1 is never selected (an empty segment), and segment lengths are
    not multiples of 32 (zero-padded tail blocks).

Where a later GEMM must read a computed operand exactly (the dgrad2 cases,
observed through the GEMMs after it), mantissas are kept to 1 or 2 bits so
that the sums stay within E4M3's 4 bits.
"""
from __future__ import annotations

import numpy as np

HI, LO = 0.0, -20.0  # the two binade bands (2^0 and 2^-20)


def _band(rng, shape, exps, axis, mmax=15, positive=False):
    """+-m * 2^exps[i], i the index along `axis`, m uniform in 1..mmax."""
    m = rng.integers(1, mmax + 1, size=shape).astype(np.float64)
    if not positive:
        m *= rng.choice([-1.0, 1.0], size=shape)
    e = np.asarray(exps, np.float64)
    shp = [1] * len(shape)
    shp[axis] = shape[axis]
    return m * np.exp2(e.reshape(shp))


def _alt(n, a=HI, b=LO):
    return np.where(np.arange(n) % 2 == 0, a, b)


def equal_pair_logits(T, E):
    """Token t selects two experts with equal logits (gates exactly 1/2):
    (0,1), (1,2), (0,2) in turn; expert E-1 (E >= 4) is never selected."""
    lg = np.full((T, E), -50.0)
    pairs = [(0, 1), (1, 2), (0, 2)]
    for t in range(T):
        a, b = pairs[t % 3]
        lg[t, a] = lg[t, b] = 0.0
    return lg


def _one_hot(T, d, cols, vals):
    x = np.zeros((T, d))
    x[np.arange(T), cols] = vals
    return x


# For each case: the GEMM it targets, and per operand of that GEMM the output
# (a key of the MXFP8 layer oracle's result) in which a blocking along the
# wrong axis shows, and whether it shows per output row ("row": the operand's
# band follows the output's rows) or per output column ("col").
TARGETS = {
    "gemm1": ("GEMM1", [("x rows along d", "hg", "row"), ("w_gate, w_up columns along d", "hg", "col")]),
    "gemm2": ("GEMM2", [("a rows along f", "ye", "row"), ("w_down columns along f", "ye", "col")]),
    "dgrad2_w": ("GEMM2 dgrad", [("w_down rows along d", "dh", "col")]),
    "dgrad2_dy": ("GEMM2 dgrad", [("dy_perm rows along d", "dh", "row")]),
    "wgrad2": ("GEMM2 wgrad", [("a along the expert's rows", "dw_down", "row"),
                               ("dy_perm along the expert's rows", "dw_down", "col")]),
    "dgrad1": ("GEMM1 dgrad", [("dh rows along 2f", "dx_perm", "row"),
                               ("w_gate, w_up rows along f", "dx_perm", "col")]),
    "wgrad1": ("GEMM1 wgrad", [("x_perm along the expert's rows", "dw_gate", "row"),
                               ("dh along the expert's rows", "dw_gate", "col")]),
}


def case(name, T=100, d=128, f=128, E=4, seed=0):
    """Inputs (fp64 arrays, exactly representable in bf16) for the named case:
    dict(x, w_r, w_gate, w_up, w_down, dy, logits, k)."""
    rng = np.random.default_rng(seed + 1000 * list(TARGETS).index(name))
    t = np.arange(T)
    w_r = _band(rng, (d, E), np.full(E, -6.0), 1, mmax=3)
    lg = equal_pair_logits(T, E)
    if name == "gemm1":
        x = _band(rng, (T, d), _alt(T), 0)                 # band by token
        wg = _band(rng, (E, d, f), _alt(f) - 3, 2)          # band by output column
        wu = _band(rng, (E, d, f), _alt(f) - 3, 2)
        wd = _band(rng, (E, f, d), np.full(d, -4.0), 2)
        dy = _band(rng, (T, d), np.zeros(T), 0)
    elif name == "gemm2":
        px = np.where(t % 2 == 0, 0.0, 10.0)
        x = _one_hot(T, d, t % d, np.exp2(px))               # h_g = m 2^(6+px), h_u = +-2^px
        wg = _band(rng, (E, d, f), np.full(f, 6.0), 2, positive=True)
        wu = _band(rng, (E, d, f), np.zeros(f), 2, mmax=1)
        wd = _band(rng, (E, f, d), _alt(d), 2)              # band by output column
        dy = _band(rng, (T, d), np.zeros(T), 0)
    elif name == "dgrad2_w":
        x = _one_hot(T, d, t % d, np.ones(T))
        wg = np.full((E, d, f), 64.0)                        # h_g = 64: dh_u = 64 da
        wu = _band(rng, (E, d, f), np.zeros(f), 2, mmax=1)  # h_u = +-1
        wd = _band(rng, (E, f, d), _alt(f), 1)              # band by row (f index)
        dy = _one_hot(T, d, (3 * t) % d, rng.choice([-1.0, 1.0], T))
    elif name == "dgrad2_dy":
        x = _one_hot(T, d, t % d, np.ones(T))
        wg = np.full((E, d, f), 64.0)
        wu = _band(rng, (E, d, f), np.zeros(f), 2, mmax=1)
        wd = _band(rng, (E, f, d), np.zeros(d), 2, mmax=2)  # 1-2 bit mantissas: da stays exact
        dy = np.zeros((T, d))  # two entries per token, band by token; each column meets both bands
        p = np.exp2(_alt(T))
        dy[t, (t // 2) % 8] = rng.choice([-1.0, 1.0], T) * p
        dy[t, 8 + (t // 2) % 8] = rng.choice([-1.0, 1.0], T) * p
    elif name == "wgrad2":
        x = _one_hot(T, d, t % d, np.ones(T))
        wg = _band(rng, (E, d, f), np.full(f, 6.0), 2, positive=True)
        wu = _band(rng, (E, d, f), _alt(f), 2, mmax=1)      # a = +-m 2^(6 + band(n)): band by column
        wd = _band(rng, (E, f, d), np.full(d, -4.0), 2)
        dy = _band(rng, (T, d), _alt(d), 1)                 # band by column
    elif name == "dgrad1":
        c1 = 2 * (t % (d // 2))                             # x uses even rows of the weights only
        x = _one_hot(T, d, c1, np.ones(T))
        rows = np.where(np.arange(d) % 2 == 0, 6.0, -24.0)  # w_gate band by row (d index)
        wg = _band(rng, (E, d, f), rows, 1, positive=True)
        wu = _band(rng, (E, d, f), rows - 6.0, 1, mmax=1)
        wd = _band(rng, (E, f, d), np.zeros(d), 2, mmax=1)  # +-1
        dy = _one_hot(T, d, (5 * t) % d, rng.choice([-1.0, 1.0], T) * np.exp2(_alt(T)))  # band by token
    elif name == "wgrad1":
        c1 = 2 * (t % (d // 2))
        c2 = 2 * ((7 * t) % (d // 2)) + 1
        x = _one_hot(T, d, c1, np.ones(T))
        x[t, c2] = rng.integers(1, 16, T) * rng.choice([-1.0, 1.0], T) * np.exp2(LO)  # band by column
        odd = np.arange(d) % 2 == 1
        wg = _band(rng, (E, d, f), np.full(f, 6.0), 2, positive=True)
        wu = _band(rng, (E, d, f), np.zeros(f), 2, mmax=1)
        wg[:, odd, :] = 0.0                                 # the tiny x columns meet zero weights
        wu[:, odd, :] = 0.0
        wd = _band(rng, (E, f, d), _alt(f), 1, mmax=1)      # da = +-2^band(n) / 2: band by column of dh
        dy = _one_hot(T, d, (3 * t) % d, rng.choice([-1.0, 1.0], T))
    else:
        raise KeyError(name)
    return dict(x=x, w_r=w_r, w_gate=wg, w_up=wu, w_down=wd, dy=dy, logits=lg, k=2)
