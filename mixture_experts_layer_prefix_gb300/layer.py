"""The MoE layer's forward and backward as a sequence of libmoe calls.

This module holds device buffers (torch tensors, allocated once per shape)
and calls the C ABI in order; every step of the computation runs in the
library's kernels. Order of calls:

  forward : moe_route -> moe_permute -> moe_grouped_mlp_fwd -> moe_combine_fwd
  backward: moe_combine_bwd -> moe_route_bwd -> moe_grouped_mlp_bwd
            -> moe_permute_bwd (adds the router's share of dx)

On the MXFP8 path the dispatched activations are row-quantised where they are
produced (mx_pre, default on): moe_permute_mxfp8 writes x_perm's E4M3 rows
next to the bf16 dispatch and moe_combine_bwd_mxfp8 dy_perm's; moe_mxfp8_prepare_weights quantises every
weight once per step in both K layouts; moe_mxfp8_mlp_fwd also writes A
quantised along the experts' rows (a_cols) from its GEMM1 epilogue;
moe_mxfp8_mlp_fwd / moe_mxfp8_mlp_bwd then run no quantisation of their own
for those operands.

With fused=True (bf16 only) moe_dispatch_mlp_fwd / moe_dispatch_mlp_bwd
replace moe_permute and the two grouped-MLP calls: GEMM1 and its weight
gradient gather x's rows with TMA row gathers and x_perm is not written. The
results are bit-identical, but on GB300 the row gathers (re-issued for every
output-column tile) run far below the rate of whole-box loads, so the default
is the permute followed by box loads.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import _native as N


@dataclasses.dataclass
class Params:
    x: torch.Tensor
    w_router: torch.Tensor      # [E, d]
    bias: torch.Tensor | None   # [E] fp32
    w_gate: torch.Tensor        # [E, d, f]
    w_up: torch.Tensor          # [E, d, f]
    w_down: torch.Tensor        # [E, f, d]
    dy: torch.Tensor            # [T, d]


def torch_dtype(dtype: int):
    return torch.float32 if dtype == N.MOE_F32 else torch.bfloat16


def to_device(a: np.ndarray, dtype: int, device="cuda") -> torch.Tensor:
    """float32 numpy (bf16-exact when dtype is bf16) -> device tensor of the storage type."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device=device).to(torch_dtype(dtype))


def params_from_inputs(inp, dtype: int, device="cuda") -> Params:
    """Upload seeded synthetic inputs (synth.Inputs); w_r is stored [E, d]."""
    s = inp.s
    b = inp.bias()
    wg = torch.empty((s.E, s.d, s.f), dtype=torch_dtype(dtype), device=device)
    wu = torch.empty_like(wg)
    wd = torch.empty((s.E, s.f, s.d), dtype=torch_dtype(dtype), device=device)
    for e in range(s.E):  # expert by expert: bounded host memory for large layers
        wg[e].copy_(torch.from_numpy(inp.w_gate_e(e)))
        wu[e].copy_(torch.from_numpy(inp.w_up_e(e)))
        wd[e].copy_(torch.from_numpy(inp.w_down_e(e)))
    return Params(
        x=to_device(inp.x(), dtype, device),
        w_router=to_device(np.ascontiguousarray(inp.w_r().T), dtype, device),
        bias=None if b is None else torch.from_numpy(b).to(device),
        w_gate=wg, w_up=wu, w_down=wd,
        dy=to_device(inp.dy(), dtype, device),
    )


class Buffers:
    """Every activation, gradient and metadata buffer of one layer shape."""

    def __init__(self, T, d, E, k, f, dtype, device="cuda"):
        self.T, self.d, self.E, self.k, self.f, self.dtype = T, d, E, k, f, dtype
        R = T * k
        self.R = R
        td = torch_dtype(dtype)
        i32, f32 = torch.int32, torch.float32
        z = lambda *sh, dt=td: torch.empty(sh, dtype=dt, device=device)  # noqa: E731
        self.logits = z(T, E, dt=f32)
        self.topk_idx = z(T, k, dt=i32)
        self.gates = z(T, k, dt=f32)
        self.counts = z(E, dt=i32)
        self.offsets = z(E + 1, dt=i32)
        self.dest_row = z(T, k, dt=i32)
        self.src_row = z(R, dt=i32)
        self.x_perm = z(R, d)
        self.h_save = z(R, 2 * f)
        self.a_save = z(R, f)
        self.y_perm = z(R, d)
        self.y = z(T, d)
        self.dy_perm = z(R, d)
        self.dgates = z(T, k, dt=f32)
        self.dlogits = z(T, E, dt=f32)
        self.dw_router = z(E, d, dt=f32)
        self.dx_perm = z(R, d)
        self.dx = z(T, d)
        self.dw_gate = z(E, d, f)
        self.dw_up = z(E, d, f)
        self.dw_down = z(E, f, d)
        self.workspace = torch.empty(max(1, N.moe_workspace_size(T, d, E, k, f, dtype)),
                                     dtype=torch.uint8, device=device)
        if dtype == N.MOE_MXFP8:  # rows quantised before the dispatch / by the combine backward
            u8 = torch.uint8
            nsc = max(1, N.moe_mxfp8_row_scales_size(R, E, d))  # scale chunks by per-expert row tiles
            self.x_q, self.x_sc = z(R, d, dt=u8), z(nsc, dt=u8)
            self.dy_q, self.dy_sc = z(R, d, dt=u8), z(nsc, dt=u8)
            # the weights quantised once per step in both K layouts
            self.wq = torch.empty(max(1, N.moe_mxfp8_weights_size(E, d, f)), dtype=u8, device=device)
            # A quantised along the experts' rows by GEMM1's epilogue, read by the GEMM2 wgrad
            self.a_cols = torch.empty(max(1, N.moe_mxfp8_col_operand_size(R, E, f)), dtype=u8, device=device)


def route_stats(b: Buffers, stream=None):
    """Routing load statistics of the last moe_route into ``b``: (probs_mean [E],
    stats [4]) device tensors -- see moe_route_stats in include/moe.h."""
    pm = torch.empty(b.E, dtype=torch.float32, device=b.logits.device)
    st = torch.empty(4, dtype=torch.float32, device=b.logits.device)
    N.moe_route_stats(b.logits, b.counts, b.T, b.E, b.k, pm, st, b.workspace, stream)
    return pm, st


def fused_default(dtype: int) -> bool:
    """Whether the layer fuses the dispatch into the expert GEMMs by default:
    no (measured slower than moe_permute + box loads at every tested shape)."""
    return False


def forward(p: Params, b: Buffers, logits_in: bool = False, stream=None, fused=None, mx_pre=True):
    T, d, E, k, f, dt = b.T, b.d, b.E, b.k, b.f, b.dtype
    N.moe_route(p.x, p.w_router, p.bias, dt, T, d, E, k, b.logits,
                N.MOE_ROUTE_LOGITS_IN if logits_in else 0, b.topk_idx, b.gates, b.counts, b.offsets,
                b.dest_row, b.src_row, b.workspace, stream)
    if dt == N.MOE_MXFP8 and mx_pre:
        N.moe_mxfp8_prepare_weights(p.w_gate, p.w_up, p.w_down, E, d, f, b.wq, stream)
        N.moe_permute_mxfp8(p.x, T, d, k, E, b.dest_row, b.topk_idx, b.offsets, b.x_q, b.x_sc, b.x_perm, stream)
        N.moe_mxfp8_mlp_fwd(b.x_q, b.x_sc, b.wq, b.offsets, b.R, E, d, f, b.h_save, b.a_save, b.y_perm, b.a_cols,
                            b.workspace, stream)
    elif fused_default(dt) if fused is None else fused:
        N.moe_dispatch_mlp_fwd(p.x, b.src_row, T, k, p.w_gate, p.w_up, p.w_down, dt, b.offsets, E, d, f,
                               b.h_save, b.a_save, b.y_perm, stream)
    else:
        N.moe_permute(p.x, dt, T, d, k, b.dest_row, b.x_perm, stream)
        N.moe_grouped_mlp_fwd(b.x_perm, p.w_gate, p.w_up, p.w_down, dt, b.offsets, b.R, E, d, f, b.h_save,
                              b.a_save, b.y_perm, b.workspace, stream)
    N.moe_combine_fwd(b.y_perm, b.gates, b.dest_row, dt, T, d, k, b.y, stream)


def backward(p: Params, b: Buffers, stream=None, fused=None, mx_pre=True):
    T, d, E, k, f, dt = b.T, b.d, b.E, b.k, b.f, b.dtype
    mx = dt == N.MOE_MXFP8 and mx_pre
    if mx:
        N.moe_combine_bwd_mxfp8(p.dy, b.y_perm, b.gates, b.dest_row, b.topk_idx, b.offsets, T, d, k, E, b.dy_q,
                                b.dy_sc, b.dy_perm, b.dgates, stream)
    else:
        N.moe_combine_bwd(p.dy, b.y_perm, b.gates, b.dest_row, dt, T, d, k, b.dy_perm, b.dgates, stream)
    N.moe_route_bwd(b.dgates, b.gates, b.topk_idx, b.offsets, b.src_row, p.x, dt, T, d, E, k,
                    b.dlogits, b.dw_router, stream)
    if mx:
        N.moe_mxfp8_mlp_bwd(b.dy_q, b.dy_sc, b.dy_perm, b.x_perm, b.h_save, b.a_save, b.a_cols, b.wq, b.offsets, b.R,
                            E, d, f, b.dx_perm, b.dw_gate, b.dw_up, b.dw_down, b.workspace, stream)
    elif fused_default(dt) if fused is None else fused:
        N.moe_dispatch_mlp_bwd(b.dy_perm, p.x, b.src_row, T, k, b.h_save, b.a_save, p.w_gate, p.w_up, p.w_down,
                               dt, b.offsets, E, d, f, b.dx_perm, b.dw_gate, b.dw_up, b.dw_down, b.workspace,
                               stream)
    else:
        N.moe_grouped_mlp_bwd(b.dy_perm, b.x_perm, b.h_save, b.a_save, p.w_gate, p.w_up, p.w_down, dt,
                              b.offsets, b.R, E, d, f, b.dx_perm, b.dw_gate, b.dw_up, b.dw_down, b.workspace,
                              stream)
    N.moe_permute_bwd(b.dx_perm, dt, T, d, E, k, b.dest_row, b.topk_idx, b.dlogits, p.w_router, b.dx,
                      stream)


def step(p: Params, b: Buffers, stream=None):
    """One forward+backward pass of the layer."""
    forward(p, b, stream=stream)
    backward(p, b, stream=stream)


class HostPipeline:
    """Forward+backward over a sequence of host batches with the copies hidden.

    Every step's x and dy come from pinned host memory and its y and dx go back
    to pinned host memory. While step i computes on the caller's stream, step
    i+1's inputs travel host->device on one copy stream and step i-1's outputs
    travel device->host on another. The device inputs (x, dy) and outputs
    (y, dx) are double-buffered; every other buffer of `b` is reused by each
    step in turn, which the compute stream orders. After `run`, `p.x`, `p.dy`,
    `b.y` and `b.dx` refer to the buffers of the last step.
    """

    def __init__(self, p: Params, b: Buffers):
        self.p, self.b = p, b
        self.xin = [p.x, torch.empty_like(p.x)]
        self.dyin = [p.dy, torch.empty_like(p.dy)]
        self.yout = [b.y, torch.empty_like(b.y)]
        self.dxout = [b.dx, torch.empty_like(b.dx)]
        dev = p.x.device
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.loaded = [torch.cuda.Event(), torch.cuda.Event()]    # slot's inputs are on the device
        self.computed = [torch.cuda.Event(), torch.cuda.Event()]  # slot's step finished
        self.drained = [torch.cuda.Event(), torch.cuda.Event()]   # slot's outputs are on the host

    def run(self, xs, dys, ys, dxs, stream=None):
        """xs, dys: pinned host inputs [T, d] per step; ys, dxs: pinned host
        outputs [T, d] per step (written when the caller's stream reaches the
        end of this call)."""
        comp = stream if stream is not None else torch.cuda.current_stream()
        p, b = self.p, self.b
        n = len(xs)
        used = [False, False]
        self.h2d.wait_stream(comp)
        self.d2h.wait_stream(comp)

        def load(i):
            s = i % 2
            with torch.cuda.stream(self.h2d):
                if used[s]:
                    self.h2d.wait_event(self.computed[s])
                self.xin[s].copy_(xs[i], non_blocking=True)
                self.dyin[s].copy_(dys[i], non_blocking=True)
                self.loaded[s].record(self.h2d)

        if n:
            load(0)
        for i in range(n):
            s = i % 2
            if i + 1 < n:
                load(i + 1)
            comp.wait_event(self.loaded[s])
            if used[s]:
                comp.wait_event(self.drained[s])
            p.x, p.dy, b.y, b.dx = self.xin[s], self.dyin[s], self.yout[s], self.dxout[s]
            forward(p, b, stream=comp)
            backward(p, b, stream=comp)
            self.computed[s].record(comp)
            used[s] = True
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.computed[s])
                ys[i].copy_(self.yout[s], non_blocking=True)
                dxs[i].copy_(self.dxout[s], non_blocking=True)
                self.drained[s].record(self.d2h)
        comp.wait_stream(self.d2h)
        comp.wait_stream(self.h2d)
