"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here has the name of the C entry point it calls and takes
torch tensors (device memory owned by the caller) or None; it passes their
data pointers and the current CUDA stream, and raises MoEError on a non-zero
status. There is no fallback: if libmoe.so is missing or a call fails, the
call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_F32, MOE_BF16, MOE_MXFP8 = 0, 1, 2
MOE_ROUTE_LOGITS_IN = 1
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ALIGNMENT",
          4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE_INDEX", 7: "MOE_ERR_TIMEOUT",
          8: "MOE_ERR_DEVICE_PAIR"}

# every symbol include/moe.h declares
EXPORTS = ("moe_workspace_size", "moe_route", "moe_permute", "moe_permute_bwd", "moe_combine_fwd",
           "moe_combine_bwd", "moe_route_bwd", "moe_grouped_mlp_fwd", "moe_grouped_mlp_bwd",
           "mxfp8_quantize", "moe_get_device_error", "moe_sm_count", "moe_launch_count", "moe_route_noalloc",
           "moe_dispatch_mlp_fwd", "moe_dispatch_mlp_bwd", "moe_route_stats", "moe_permute_mxfp8",
           "moe_combine_bwd_mxfp8", "moe_mxfp8_mlp_fwd", "moe_mxfp8_mlp_bwd", "moe_mxfp8_weights_size",
           "moe_mxfp8_prepare_weights", "moe_mxfp8_row_scales_size", "moe_timing_arm", "moe_timing_finish",
           "moe_timing_read", "moe_selftest_wait_timeout", "moe_mxfp8_col_operand_size",
           "moe_use_cta_pairs")


class MoEError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load libmoe.so (build it first with the package's build module)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe.so not built ({path}); run mixture_experts_layer_prefix_gb300.build")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "moe_workspace_size": ([I, I, I, I, I, I], Z),
        "moe_route": ([P, P, P, I, I, I, I, I, P, I, P, P, P, P, P, P, P, Z, P], I),
        "moe_permute": ([P, I, I, I, I, P, P, P], I),
        "moe_permute_bwd": ([P, I, I, I, I, I, P, P, P, P, P, P], I),
        "moe_combine_fwd": ([P, P, P, I, I, I, I, P, P], I),
        "moe_combine_bwd": ([P, P, P, P, I, I, I, I, P, P, P], I),
        "moe_route_bwd": ([P, P, P, P, P, P, I, I, I, I, I, P, P, P], I),
        "moe_grouped_mlp_fwd": ([P, P, P, P, I, P, I, I, I, I, P, P, P, P, Z, P], I),
        "moe_grouped_mlp_bwd": ([P, P, P, P, P, P, P, I, P, I, I, I, I, P, P, P, P, P, Z, P], I),
        "mxfp8_quantize": ([P, I, I, I, P, I, P, P, P], I),
        "moe_get_device_error": ([P], I),
        "moe_sm_count": ([], I),
        "moe_launch_count": ([], ctypes.c_uint64),
        "moe_route_noalloc": ([P, P, P, I, I, I, I, I, P, I, P, P, P, P, P, P, P], I),
        "moe_dispatch_mlp_fwd": ([P, P, I, I, P, P, P, I, P, I, I, I, P, P, P, P], I),
        "moe_route_stats": ([P, P, I, I, I, P, P, P, Z, P], I),
        "moe_permute_mxfp8": ([P, I, I, I, I, P, P, P, P, P, P, P], I),
        "moe_combine_bwd_mxfp8": ([P, P, P, P, P, P, I, I, I, I, P, P, P, P, P], I),
        "moe_mxfp8_row_scales_size": ([I, I, I], Z),
        "moe_mxfp8_mlp_fwd": ([P, P, P, P, I, I, I, I, P, P, P, P, P, Z, P], I),
        "moe_mxfp8_mlp_bwd": ([P, P, P, P, P, P, P, P, P, I, I, I, I, P, P, P, P, P, Z, P], I),
        "moe_mxfp8_col_operand_size": ([I, I, I], Z),
        "moe_mxfp8_weights_size": ([I, I, I], Z),
        "moe_mxfp8_prepare_weights": ([P, P, P, I, I, I, P, Z, P], I),
        "moe_dispatch_mlp_bwd": ([P, P, P, I, I, P, P, P, P, P, I, P, I, I, I, P, P, P, P, P, Z, P], I),
        "moe_timing_arm": ([I], I),
        "moe_timing_finish": ([P], I),
        "moe_timing_read": ([P, P, I], I),
        "moe_selftest_wait_timeout": ([ctypes.c_longlong, P, P], I),
        "moe_use_cta_pairs": ([I], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _chk(fn, code):
    if code != 0:
        raise MoEError(fn, code)


def moe_workspace_size(T, d, E, k, f, dtype):
    return int(load().moe_workspace_size(T, d, E, k, f, dtype))


def moe_route(x, w_router, bias, dtype, T, d, E, k, logits, flags, topk_idx, gates, counts, offsets,
              dest_row, src_row, workspace, stream=None):
    _chk("moe_route", load().moe_route(_p(x), _p(w_router), _p(bias), dtype, T, d, E, k, _p(logits),
                                       flags, _p(topk_idx), _p(gates), _p(counts), _p(offsets),
                                       _p(dest_row), _p(src_row), _p(workspace), _nbytes(workspace),
                                       _s(stream)))


def moe_permute(x, dtype, T, d, k, dest_row, x_perm, stream=None):
    _chk("moe_permute", load().moe_permute(_p(x), dtype, T, d, k, _p(dest_row), _p(x_perm), _s(stream)))


def moe_permute_bwd(dx_perm, dtype, T, d, E, k, dest_row, topk_idx, dlogits, w_router, dx, stream=None):
    _chk("moe_permute_bwd", load().moe_permute_bwd(_p(dx_perm), dtype, T, d, E, k, _p(dest_row),
                                                   _p(topk_idx), _p(dlogits), _p(w_router), _p(dx),
                                                   _s(stream)))


def moe_combine_fwd(y_perm, gates, dest_row, dtype, T, d, k, y, stream=None):
    _chk("moe_combine_fwd", load().moe_combine_fwd(_p(y_perm), _p(gates), _p(dest_row), dtype, T, d, k,
                                                   _p(y), _s(stream)))


def moe_combine_bwd(dy, y_perm, gates, dest_row, dtype, T, d, k, dy_perm, dgates, stream=None):
    _chk("moe_combine_bwd", load().moe_combine_bwd(_p(dy), _p(y_perm), _p(gates), _p(dest_row), dtype, T,
                                                   d, k, _p(dy_perm), _p(dgates), _s(stream)))


def moe_route_bwd(dgates, gates, topk_idx, offsets, src_row, x, dtype, T, d, E, k, dlogits,
                  dw_router, stream=None):
    _chk("moe_route_bwd", load().moe_route_bwd(_p(dgates), _p(gates), _p(topk_idx), _p(offsets),
                                               _p(src_row), _p(x), dtype, T, d, E, k, _p(dlogits),
                                               _p(dw_router), _s(stream)))


def moe_grouped_mlp_fwd(x_perm, w_gate, w_up, w_down, dtype, offsets, R, E, d, f, h_save, a_save,
                        y_perm, workspace, stream=None):
    _chk("moe_grouped_mlp_fwd", load().moe_grouped_mlp_fwd(
        _p(x_perm), _p(w_gate), _p(w_up), _p(w_down), dtype, _p(offsets), R, E, d, f, _p(h_save),
        _p(a_save), _p(y_perm), _p(workspace), _nbytes(workspace), _s(stream)))


def moe_grouped_mlp_bwd(dy_perm, x_perm, h_save, a_save, w_gate, w_up, w_down, dtype, offsets, R, E, d,
                        f, dx_perm, dw_gate, dw_up, dw_down, workspace, stream=None):
    _chk("moe_grouped_mlp_bwd", load().moe_grouped_mlp_bwd(
        _p(dy_perm), _p(x_perm), _p(h_save), _p(a_save), _p(w_gate), _p(w_up), _p(w_down), dtype,
        _p(offsets), R, E, d, f, _p(dx_perm), _p(dw_gate), _p(dw_up), _p(dw_down), _p(workspace),
        _nbytes(workspace), _s(stream)))


def mxfp8_quantize(src, rows, K, axis, seg_offsets, nseg, dst_e4m3, dst_e8m0, stream=None):
    _chk("mxfp8_quantize", load().mxfp8_quantize(_p(src), rows, K, axis, _p(seg_offsets), nseg,
                                                 _p(dst_e4m3), _p(dst_e8m0), _s(stream)))


def moe_get_device_error(stream=None):
    return int(load().moe_get_device_error(_s(stream)))


def moe_sm_count():
    return int(load().moe_sm_count())


def moe_launch_count():
    return int(load().moe_launch_count())


def moe_route_noalloc(x, w_router, bias, dtype, T, d, E, k, logits, flags, topk_idx, gates, counts, offsets,
                      dest_row, src_row, stream=None):
    """moe_route without a workspace argument: for callers that cannot allocate."""
    _chk("moe_route_noalloc", load().moe_route_noalloc(
        _p(x), _p(w_router), _p(bias), dtype, T, d, E, k, _p(logits), flags, _p(topk_idx), _p(gates),
        _p(counts), _p(offsets), _p(dest_row), _p(src_row), _s(stream)))


def moe_dispatch_mlp_fwd(x, src_row, T, k, w_gate, w_up, w_down, dtype, offsets, E, d, f, h_save, a_save,
                         y_perm, stream=None):
    _chk("moe_dispatch_mlp_fwd", load().moe_dispatch_mlp_fwd(
        _p(x), _p(src_row), T, k, _p(w_gate), _p(w_up), _p(w_down), dtype, _p(offsets), E, d, f, _p(h_save),
        _p(a_save), _p(y_perm), _s(stream)))


def moe_dispatch_mlp_bwd(dy_perm, x, src_row, T, k, h_save, a_save, w_gate, w_up, w_down, dtype, offsets, E, d,
                         f, dx_perm, dw_gate, dw_up, dw_down, workspace, stream=None):
    _chk("moe_dispatch_mlp_bwd", load().moe_dispatch_mlp_bwd(
        _p(dy_perm), _p(x), _p(src_row), T, k, _p(h_save), _p(a_save), _p(w_gate), _p(w_up), _p(w_down), dtype,
        _p(offsets), E, d, f, _p(dx_perm), _p(dw_gate), _p(dw_up), _p(dw_down), _p(workspace), _nbytes(workspace),
        _s(stream)))


def moe_route_stats(logits, counts, T, E, k, probs_mean, stats, workspace, stream=None):
    _chk("moe_route_stats", load().moe_route_stats(_p(logits), _p(counts), T, E, k, _p(probs_mean), _p(stats),
                                                   _p(workspace), _nbytes(workspace), _s(stream)))


def moe_mxfp8_row_scales_size(R, E, K):
    return load().moe_mxfp8_row_scales_size(R, E, K)


def moe_permute_mxfp8(x, T, d, k, E, dest_row, topk_idx, offsets, x_codes, x_scales, x_perm=None, stream=None):
    _chk("moe_permute_mxfp8", load().moe_permute_mxfp8(_p(x), T, d, k, E, _p(dest_row), _p(topk_idx), _p(offsets),
                                                       _p(x_codes), _p(x_scales), _p(x_perm), _s(stream)))


def moe_combine_bwd_mxfp8(dy, y_perm, gates, dest_row, topk_idx, offsets, T, d, k, E, dy_codes, dy_scales, dy_perm,
                          dgates, stream=None):
    _chk("moe_combine_bwd_mxfp8", load().moe_combine_bwd_mxfp8(
        _p(dy), _p(y_perm), _p(gates), _p(dest_row), _p(topk_idx), _p(offsets), T, d, k, E, _p(dy_codes),
        _p(dy_scales), _p(dy_perm), _p(dgates), _s(stream)))


def moe_mxfp8_weights_size(E, d, f):
    return load().moe_mxfp8_weights_size(E, d, f)


def moe_mxfp8_prepare_weights(w_gate, w_up, w_down, E, d, f, wq, stream=None):
    _chk("moe_mxfp8_prepare_weights", load().moe_mxfp8_prepare_weights(
        _p(w_gate), _p(w_up), _p(w_down), E, d, f, _p(wq), _nbytes(wq), _s(stream)))


def moe_mxfp8_col_operand_size(R, E, K):
    return load().moe_mxfp8_col_operand_size(R, E, K)


def moe_mxfp8_mlp_fwd(x_codes, x_scales, wq, offsets, R, E, d, f, h_save, a_save, y_perm, a_cols, workspace,
                      stream=None):
    _chk("moe_mxfp8_mlp_fwd", load().moe_mxfp8_mlp_fwd(
        _p(x_codes), _p(x_scales), _p(wq), _p(offsets), R, E, d, f, _p(h_save), _p(a_save), _p(y_perm), _p(a_cols),
        _p(workspace), _nbytes(workspace), _s(stream)))


def moe_mxfp8_mlp_bwd(dy_codes, dy_scales, dy_perm, x_perm, h_save, a_save, a_cols, wq, offsets, R, E, d, f, dx_perm,
                      dw_gate, dw_up, dw_down, workspace, stream=None):
    _chk("moe_mxfp8_mlp_bwd", load().moe_mxfp8_mlp_bwd(
        _p(dy_codes), _p(dy_scales), _p(dy_perm), _p(x_perm), _p(h_save), _p(a_save), _p(a_cols), _p(wq),
        _p(offsets), R, E, d, f, _p(dx_perm), _p(dw_gate), _p(dw_up), _p(dw_down), _p(workspace), _nbytes(workspace),
        _s(stream)))


def moe_timing_arm(n):
    _chk("moe_timing_arm", load().moe_timing_arm(int(n)))


def moe_timing_finish(stream=None):
    _chk("moe_timing_finish", load().moe_timing_finish(_s(stream)))


def moe_timing_read(cap=256):
    """[(kernel name, ms)] of the launches recorded since moe_timing_arm."""
    ms = (ctypes.c_float * cap)()
    names = (ctypes.c_char_p * cap)()
    n = load().moe_timing_read(ms, names, cap)
    if n < 0:
        raise MoEError("moe_timing_read", 1)
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


def moe_use_cta_pairs(enable):
    _chk("moe_use_cta_pairs", load().moe_use_cta_pairs(1 if enable else 0))


def moe_selftest_wait_timeout(cycles, out, stream=None):
    _chk("moe_selftest_wait_timeout", load().moe_selftest_wait_timeout(int(cycles), _p(out), _s(stream)))
