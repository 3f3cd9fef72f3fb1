"""fp64 CPU oracle for the single-GPU MoE layer -- TEST INFRASTRUCTURE.

This package is the plain, slow definition that the CUDA library is checked
against. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import it; the library never does.

The arithmetic lives in ``moe_oracle.c`` (plain C, every operation in double);
this module compiles it with gcc on first use and exposes numpy-level calls.
Each function cites what it follows:

* "Introducing Olmo-core 3", section "Scaling and optimizing MoE training":
  routing to experts, placement of routed rows into per-expert input buffers,
  routing metadata kept on the device, grouped expert GEMMs, MXFP8.
* The benchmark workload's own definition (8- vs 128-expert top-4 layer):
  softmax over E, top-k, renormalised gates, SwiGLU experts, E4M3 elements
  with one E8M0 scale per 32 along K.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(brute force, library special cases, finite differences, spec tables).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so next to it (gcc, -O2, portable flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oc_router_logits.argtypes = [P, P, P, I, I, I, P, I]
            lib.oc_topk.argtypes = [P, I, I, I, P]
            lib.oc_gates.argtypes = [P, P, I, I, I, P]
            lib.oc_route_stats.argtypes = [P, P, I, I, I, P, P]
            lib.oc_dispatch.argtypes = [P, I, I, I, P, P, P, P]
            lib.oc_forward.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, I]
            lib.oc_backward.argtypes = [P] * 12 + [I] * 5 + [P] * 10 + [I]
            lib.oc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oc_e4m3_decode.restype = ctypes.c_double
            lib.oc_e4m3_encode.argtypes = [ctypes.c_double]
            lib.oc_e4m3_encode.restype = ctypes.c_uint8
            lib.oc_e8m0_exponent.argtypes = [ctypes.c_double]
            lib.oc_e8m0_exponent.restype = ctypes.c_int
            lib.oc_mxfp8_quantize_rows.argtypes = [P, ctypes.c_long, ctypes.c_long, P, P]
            lib.oc_mxfp8_quantize_cols_segmented.argtypes = [P, ctypes.c_long, ctypes.c_long, P, I, P, P]
            lib.oc_mxfp8_quantize_rows_f64.argtypes = [P, ctypes.c_long, ctypes.c_long, P, P]
            lib.oc_mxfp8_quantize_cols_segmented_f64.argtypes = [P, ctypes.c_long, ctypes.c_long, P, I, P, P]
            _lib = lib
    return _lib


def _threads(n):
    return int(n) if n else (len(os.sched_getaffinity(0)) or 1)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return a.ctypes.data if a is not None else None


# --------------------------------------------------------------------- routing
def router_logits(x, w_r, bias=None, nthreads=None):
    """l[t,e] = bias[e] + x[t] . w_r[:, e] in fp64 (router GEMM of the routing step)."""
    x, w_r = _f32(x), _f32(w_r)
    T, d = x.shape
    E = w_r.shape[1]
    b = _f32(bias) if bias is not None else None
    out = np.empty((T, E), np.float64)
    _L().oc_router_logits(_p(x), _p(w_r), _p(b), T, d, E, _p(out), _threads(nthreads))
    return out


def topk(logits, k):
    """Indices of the k largest logits per token; ties keep the smaller index;
    slots ordered by (logit desc, index asc)."""
    l = _f64(logits)
    T, E = l.shape
    idx = np.empty((T, k), np.int32)
    _L().oc_topk(_p(l), T, E, k, _p(idx))
    return idx


def gates(logits, topk_idx):
    """Softmax over the selected logits (= softmax over E, renormalised over the top-k)."""
    l, idx = _f64(logits), _i32(topk_idx)
    T, E = l.shape
    k = idx.shape[1]
    g = np.empty((T, k), np.float64)
    _L().oc_gates(_p(l), _p(idx), T, E, k, _p(g))
    return g


def route_stats(logits, counts, k):
    """Routing load statistics: (probs_mean [E], stats [4]) with stats =
    (E * sum_e f_e probs_mean_e, max load / mean load, empty experts,
    std / mean of the counts), f_e = counts_e / (T k), probs_mean the mean
    full softmax over E. The pages give no formula for a balance metric: parity
    unpinned by the pages (pinned here by closed forms and invariants)."""
    l, c = _f64(logits), _i32(counts)
    T, E = l.shape
    pm = np.empty(E, np.float64)
    st = np.empty(4, np.float64)
    _L().oc_route_stats(_p(l), _p(c), T, E, k, _p(pm), _p(st))
    return pm, st


def dispatch(topk_idx, E):
    """counts[E], offsets[E+1], dest_row[T,k], src_row[T*k]: routed pair (t, j)
    goes to row dest_row[t, j] of its expert's contiguous block; rows of one
    expert follow token order (placement into expert input buffers)."""
    idx = _i32(topk_idx)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    dest = np.empty((T, k), np.int32)
    src = np.empty(T * k, np.int32)
    _L().oc_dispatch(_p(idx), T, E, k, _p(counts), _p(offsets), _p(dest), _p(src))
    return counts, offsets, dest, src


def route(logits, k, E=None):
    """Full routing step from given logits: top-k, gates and dispatch metadata."""
    l = _f64(logits)
    E = l.shape[1] if E is None else E
    idx = topk(l, k)
    g = gates(l, idx)
    counts, offsets, dest, src = dispatch(idx, E)
    return dict(topk_idx=idx, gates=g, counts=counts, offsets=offsets, dest_row=dest, src_row=src)


# ---------------------------------------------------------------- expert MLP
def forward(x, w_gate, w_up, w_down, topk_idx, gates_, nthreads=None):
    """Token-by-token SwiGLU experts and gate-weighted combine. Returns a dict
    with y [T,d] and the per-pair values hg, hu, a [T*k,f], ye [T*k,d]."""
    x, wg, wu, wd = _f32(x), _f32(w_gate), _f32(w_up), _f32(w_down)
    idx, g = _i32(topk_idx), _f64(gates_)
    T, d = x.shape
    E, _, f = wg.shape
    k = idx.shape[1]
    R = T * k
    hg = np.empty((R, f)); hu = np.empty((R, f)); a = np.empty((R, f))
    ye = np.empty((R, d)); y = np.empty((T, d))
    _L().oc_forward(_p(x), _p(wg), _p(wu), _p(wd), _p(idx), _p(g), T, d, E, k, f,
                    _p(hg), _p(hu), _p(a), _p(ye), _p(y), _threads(nthreads))
    return dict(y=y, hg=hg, hu=hu, a=a, ye=ye)


def backward(x, w_r, w_gate, w_up, w_down, dy, topk_idx, gates_, fwd, nthreads=None):
    """Backward of the layer for upstream gradient dy; returns dgates, dlogits,
    dx (expert path + router path), dw_gate, dw_up, dw_down, dw_r and the
    per-pair dye [T*k,d], dhg, dhu [T*k,f]."""
    x, wr, wg, wu, wd, dy = map(_f32, (x, w_r, w_gate, w_up, w_down, dy))
    idx, g = _i32(topk_idx), _f64(gates_)
    T, d = x.shape
    E, _, f = wg.shape
    k = idx.shape[1]
    R = T * k
    out = dict(dgates=np.empty((T, k)), dlogits=np.empty((T, E)), dx=np.empty((T, d)),
               dye=np.empty((R, d)), dhg=np.empty((R, f)), dhu=np.empty((R, f)),
               dw_gate=np.empty((E, d, f)), dw_up=np.empty((E, d, f)), dw_down=np.empty((E, f, d)),
               dw_r=np.empty((d, E)))
    _L().oc_backward(_p(x), _p(wr), _p(wg), _p(wu), _p(wd), _p(dy), _p(idx), _p(g),
                     _p(fwd["hg"]), _p(fwd["hu"]), _p(fwd["a"]), _p(fwd["ye"]),
                     T, d, E, k, f,
                     _p(out["dgates"]), _p(out["dlogits"]), _p(out["dx"]), _p(out["dye"]),
                     _p(out["dhg"]), _p(out["dhu"]), _p(out["dw_gate"]), _p(out["dw_up"]),
                     _p(out["dw_down"]), _p(out["dw_r"]), _threads(nthreads))
    return out


def layer(x, w_r, w_gate, w_up, w_down, dy, k, bias=None, logits=None, nthreads=None):
    """Whole layer forward+backward. ``logits`` (e.g. fp32 values widened) replaces
    the router GEMM when given, so routing decisions can be taken on exactly the
    logits another implementation produced."""
    E = w_gate.shape[0]
    if logits is None:
        logits = router_logits(x, w_r, bias, nthreads)
    r = route(logits, k, E)
    fw = forward(x, w_gate, w_up, w_down, r["topk_idx"], r["gates"], nthreads)
    bw = backward(x, w_r, w_gate, w_up, w_down, dy, r["topk_idx"], r["gates"], fw, nthreads)
    out = dict(logits=np.asarray(logits, np.float64))
    out.update(r); out.update(fw); out.update(bw)
    return out


# ---------------------------------------------------------------------- MXFP8
def e4m3_decode(code: int) -> float:
    return _L().oc_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return int(_L().oc_e4m3_encode(float(v)))


def e8m0_exponent(amax: float) -> int:
    return int(_L().oc_e8m0_exponent(float(amax)))


def mxfp8_quantize_rows(v):
    """[rows, K] -> (codes uint8 [rows, K], E8M0 bytes uint8 [rows, K/32]); blocks of
    32 consecutive elements along K inside each row."""
    v = _f32(v)
    rows, K = v.shape
    assert K % 32 == 0
    q = np.empty((rows, K), np.uint8)
    s = np.empty((rows, K // 32), np.uint8)
    _L().oc_mxfp8_quantize_rows(_p(v), rows, K, _p(q), _p(s))
    return q, s


def mxfp8_quantize_cols_segmented(v, seg):
    """[rows, C] quantised along rows inside each segment [seg[g], seg[g+1]):
    blocks of 32 rows start at each segment's first row and the last block of
    a segment is zero-padded. Returns codes [rows, C] and scales
    [sum_g ceil(len_g/32), C]."""
    v = _f32(v)
    seg = _i32(seg)
    rows, C = v.shape
    nblk = int(sum((int(seg[g + 1]) - int(seg[g]) + 31) // 32 for g in range(len(seg) - 1)))
    q = np.empty((rows, C), np.uint8)
    s = np.empty((max(nblk, 0), C), np.uint8)
    _L().oc_mxfp8_quantize_cols_segmented(_p(v), rows, C, _p(seg), len(seg) - 1, _p(q), _p(s))
    return q, s


_E4M3_TABLE = None


def e4m3_table():
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)], np.float64)
    return _E4M3_TABLE


def mxfp8_dequantize_rows(q, s):
    """Values = decode(code) * 2^(scale-127), blocks of 32 along the last axis."""
    vals = e4m3_table()[q]
    sc = np.ldexp(1.0, s.astype(np.int32) - 127)
    return vals * np.repeat(sc, 32, axis=1)


def mxfp8_dequantize_cols_segmented(q, s, seg):
    vals = e4m3_table()[q].copy()
    seg = np.asarray(seg)
    brow = 0
    for g in range(len(seg) - 1):
        for b0 in range(int(seg[g]), int(seg[g + 1]), 32):
            b1 = min(b0 + 32, int(seg[g + 1]))
            vals[b0:b1] *= np.ldexp(1.0, s[brow].astype(np.int32) - 127)[None, :]
            brow += 1
    return vals


def mxfp8_fakequant_rows(v):
    """dequantise(quantise(v)) with 32-element blocks along the last axis (fp64 in, fp64 out)."""
    v = _f64(v)
    rows, K = v.shape
    q = np.empty((rows, K), np.uint8)
    s = np.empty((rows, K // 32), np.uint8)
    _L().oc_mxfp8_quantize_rows_f64(_p(v), rows, K, _p(q), _p(s))
    return mxfp8_dequantize_rows(q, s)


def mxfp8_fakequant_cols_segmented(v, seg):
    """dequantise(quantise(v)) with blocks of 32 rows starting at each segment's
    first row (fp64 in, fp64 out)."""
    v = _f64(v)
    seg = _i32(seg)
    rows, C = v.shape
    nblk = int(sum((int(seg[g + 1]) - int(seg[g]) + 31) // 32 for g in range(len(seg) - 1)))
    q = np.empty((rows, C), np.uint8)
    s = np.empty((max(nblk, 0), C), np.uint8)
    _L().oc_mxfp8_quantize_cols_segmented_f64(_p(v), rows, C, _p(seg), len(seg) - 1, _p(q), _p(s))
    return mxfp8_dequantize_cols_segmented(q, s, seg)
