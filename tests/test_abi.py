"""The C ABI library: it builds, loads, exports every declared symbol, and
rejects bad arguments synchronously (no GPU needed: nothing is launched)."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_prefix_gb300 import _native as N
from mixture_experts_layer_prefix_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.load()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:moe_status|size_t|int|uint64_t)\s+(\w+)\s*\(", src, flags=re.M)
    return names


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(N.EXPORTS) <= set(names), set(N.EXPORTS) - set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_workspace_size_is_host_only(lib):
    assert N.moe_workspace_size(16384, 2048, 128, 4, 1024, N.MOE_BF16) > 0
    assert N.moe_workspace_size(-1, 2048, 128, 4, 1024, N.MOE_BF16) == 0


FAKE = 0x100000  # never dereferenced: every call below fails validation first


def test_invalid_arguments_rejected_before_launch(lib):
    L = lib
    # k > E
    assert L.moe_route(FAKE, FAKE, None, 1, 8, 64, 4, 5, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                       FAKE, 1 << 20, None) == 1
    # k > 8 and d not a multiple of 64: unsupported
    assert L.moe_route(FAKE, FAKE, None, 1, 8, 64, 16, 9, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                       FAKE, 1 << 20, None) == 2
    assert L.moe_permute(FAKE, 1, 8, 96, 2, FAKE, FAKE, None) == 2
    # misaligned pointer
    assert L.moe_permute(FAKE + 2, 1, 8, 64, 2, FAKE, FAKE, None) == 3
    # unknown dtype
    assert L.moe_combine_fwd(FAKE, FAKE, FAKE, 7, 8, 64, 2, FAKE, None) == 2
    # workspace too small
    assert L.moe_route(FAKE, FAKE, None, 1, 4096, 64, 16, 2, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE,
                       FAKE, FAKE, 16, None) == 4
    # missing buffer
    assert L.moe_combine_bwd(FAKE, None, FAKE, FAKE, 1, 8, 64, 2, FAKE, FAKE, None) == 1
    # router term: all three or none
    assert L.moe_permute_bwd(FAKE, 1, 8, 64, 4, 2, FAKE, FAKE, None, FAKE, FAKE, None) == 1
    # f not a multiple of 64
    assert L.moe_grouped_mlp_fwd(FAKE, FAKE, FAKE, FAKE, 1, FAKE, 16, 4, 64, 100, FAKE, FAKE, FAKE,
                                 FAKE, 0, None) == 2


def test_fused_dispatch_arguments_rejected_before_launch(lib):
    L = lib
    # fp32 / MXFP8 are not fused: unsupported
    assert L.moe_dispatch_mlp_fwd(FAKE, FAKE, 8, 2, FAKE, FAKE, FAKE, 0, FAKE, 4, 64, 64, FAKE, FAKE, FAKE,
                                  None) == 2
    assert L.moe_dispatch_mlp_fwd(FAKE, FAKE, 8, 2, FAKE, FAKE, FAKE, 2, FAKE, 4, 64, 64, FAKE, FAKE, FAKE,
                                  None) == 2
    # k > E
    assert L.moe_dispatch_mlp_fwd(FAKE, FAKE, 8, 5, FAKE, FAKE, FAKE, 1, FAKE, 4, 64, 64, FAKE, FAKE, FAKE,
                                  None) == 1
    # missing src_row
    assert L.moe_dispatch_mlp_fwd(FAKE, None, 8, 2, FAKE, FAKE, FAKE, 1, FAKE, 4, 64, 64, FAKE, FAKE, FAKE,
                                  None) == 1
    # T*k past the int range
    assert L.moe_dispatch_mlp_fwd(FAKE, FAKE, 1 << 30, 4, FAKE, FAKE, FAKE, 1, FAKE, 4, 64, 64, FAKE, FAKE,
                                  FAKE, None) == 2
    # backward: workspace too small for dh, misaligned x
    assert L.moe_dispatch_mlp_bwd(FAKE, FAKE, FAKE, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 4, 64, 64,
                                  FAKE, FAKE, FAKE, FAKE, FAKE, 16, None) == 4
    assert L.moe_dispatch_mlp_bwd(FAKE, FAKE + 8, FAKE, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 4, 64, 64,
                                  FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 3


def test_route_stats_arguments_rejected_before_launch(lib):
    L = lib
    assert L.moe_route_stats(FAKE, FAKE, 8, 4, 5, FAKE, FAKE, FAKE, 1 << 20, None) == 1      # k > E
    assert L.moe_route_stats(FAKE, FAKE, 8, 2048, 2, FAKE, FAKE, FAKE, 1 << 20, None) == 2   # E > 1024
    assert L.moe_route_stats(FAKE, FAKE, 4096, 128, 4, FAKE, FAKE, FAKE, 16, None) == 4      # workspace
    assert L.moe_route_stats(FAKE, None, 8, 4, 2, FAKE, FAKE, FAKE, 1 << 20, None) == 1      # counts


def test_mxfp8_dispatch_arguments_rejected_before_launch(lib):
    L = lib
    F = FAKE
    assert L.moe_permute_mxfp8(F, 8, 96, 2, 4, F, F, F, F, F, None, None) == 2            # d % 64
    assert L.moe_permute_mxfp8(F, 8, 320, 2, 4, F, F, F, F, F, None, None) == 2           # d % 128 (scale chunks)
    assert L.moe_permute_mxfp8(F, 8, 128, 2, 4, F, F, F, None, F, None, None) == 1        # codes missing
    assert L.moe_permute_mxfp8(F, 8, 128, 2, 4, F, None, F, F, F, None, None) == 1        # topk_idx missing
    assert L.moe_permute_mxfp8(F, 8, 128, 2, 4, F, F, None, F, F, None, None) == 1        # offsets missing
    assert L.moe_permute_mxfp8(F, 8, 128, 2, 4, F, F, F, F, F, F + 4, None) == 3          # x_perm aligned
    assert L.moe_permute_mxfp8(F, 8, 128, 5, 4, F, F, F, F, F, None, None) == 1           # k > E
    assert L.moe_combine_bwd_mxfp8(F, F, F, F, F, F, 8, 128, 9, 16, F, F, None, F, None) == 2  # k > 8
    assert L.moe_combine_bwd_mxfp8(F, F, F, F, F, F, 8, 320, 2, 16, F, F, None, F, None) == 2  # d % 128
    assert L.moe_combine_bwd_mxfp8(F, F, F, F, None, F, 8, 128, 2, 16, F, F, None, F, None) == 1  # topk_idx
    # scale chunks of a row operand: (R + 127 E) / 128 + 1 groups of 4 K bytes
    assert L.moe_mxfp8_row_scales_size(1000, 8, 256) == ((1000 + 127 * 8) // 128 + 1) * 4 * 256
    assert L.moe_mxfp8_row_scales_size(1000, 8, 96) == 0
    # d not a multiple of 128 for the block-scaled GEMMs
    assert L.moe_mxfp8_mlp_fwd(FAKE, FAKE, FAKE, FAKE, 16, 4, 192, 128, FAKE, FAKE, FAKE, None, FAKE, 1 << 30,
                               None) == 2
    assert L.moe_mxfp8_mlp_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 16, 4, 128, 128, FAKE, FAKE,
                               FAKE, FAKE, FAKE, 16, None) == 4                            # workspace
    # a_cols misaligned
    assert L.moe_mxfp8_mlp_fwd(FAKE, FAKE, FAKE, FAKE, 16, 4, 128, 128, FAKE, FAKE, FAKE, FAKE + 4, FAKE, 1 << 30,
                               None) == 3
    # an operand quantised along the experts' rows: codes (256-byte padded) + scale chunks
    assert L.moe_mxfp8_col_operand_size(1000, 8, 256) == 1000 * 256 + ((1000 + 127) // 128 + 8 + 1) * 256 * 4
    assert L.moe_mxfp8_col_operand_size(1000, 8, 96) == 0
    assert L.moe_mxfp8_weights_size(4, 128, 128) > 4 * 128 * 128 * 3 * 2
    assert L.moe_mxfp8_prepare_weights(FAKE, FAKE, FAKE, 4, 128, 128, FAKE, 16, None) == 4  # wq too small
    assert L.moe_mxfp8_prepare_weights(FAKE, FAKE, FAKE, 4, 192, 128, FAKE, 1 << 30, None) == 2


def test_row_scale_chunks_fit_every_routing(lib):
    """The scale-chunk layout of row operands (include/moe.h): expert e's
    128-row tiles are groups (offsets[e] + 127 e) / 128 + m. For random and
    extreme per-expert counts the groups of different experts never overlap
    and every byte of every group lies inside moe_mxfp8_row_scales_size."""
    import numpy as np
    rng = np.random.default_rng(7)
    cases = [np.full(8, 512), np.zeros(16, np.int64), np.array([0, 1, 127, 128, 129, 255, 256, 0, 1000]),
             np.array([65536] + [0] * 127)]
    cases += [rng.integers(0, 700, size=E) for E in (1, 2, 31, 128, 1024)]
    for counts in cases:
        counts = np.asarray(counts, np.int64)
        E, R = len(counts), int(counts.sum())
        offs = np.concatenate([[0], np.cumsum(counts)])
        K = 256
        size = lib.moe_mxfp8_row_scales_size(R, E, K)
        used = []
        for e in range(E):
            base = (offs[e] + 127 * e) // 128
            tiles = -(-int(counts[e]) // 128)
            used += [base + m for m in range(tiles)]
        assert len(used) == len(set(used)), counts
        if used:
            assert (max(used) + 1) * 4 * K <= size, (counts, size)
