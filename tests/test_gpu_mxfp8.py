"""MXFP8 quantisation on the GPU: codes and E8M0 scale bytes bit-exact against
the oracle's spec-derived quantiser, for blocks along rows and for blocks of
32 rows inside ragged segments (empty segments, ragged tails, zero blocks,
a wide dynamic range)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_prefix_gb300 import _native as N
from mixture_experts_layer_prefix_gb300 import build as B
from mixture_experts_layer_prefix_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    N.load()


def _values(rows, K, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((rows, K)) * np.exp(rng.uniform(-20, 20, (rows, 1)))
    v[rng.random((rows, K)) < 0.01] = 0.0
    v = synth.round_bf16(v.astype(np.float32))
    if rows > 3 and K >= 64:
        v[3, 32:64] = 0.0
        v[2, :32] = 448.0
        v[1, :32] = -450.0  # bf16-exact, just above 448
    return v


def _dev(v):
    return torch.from_numpy(v).to("cuda").to(torch.bfloat16)


@pytest.mark.parametrize("rows,K", [(1, 32), (37, 256), (1000, 2048), (4096, 1024)])
def test_quantize_rows_bit_exact(rows, K):
    v = _values(rows, K, rows + K)
    q = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    N.mxfp8_quantize(_dev(v), rows, K, 0, None, 0, q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp8_quantize_rows(v)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("seg", [[0, 5, 5, 70, 100], [0, 0, 33, 33, 64, 1000, 1001], None])
def test_quantize_segmented_columns_bit_exact(seg):
    rows = 100 if seg is None else seg[-1]
    C = 512
    v = _values(rows, C, 7)
    segs = np.array(seg if seg is not None else [0, rows], np.int32)
    nseg = len(segs) - 1
    nblk_max = (rows + 31) // 32 + nseg
    q = torch.zeros((rows, C), dtype=torch.uint8, device="cuda")
    s = torch.zeros((nblk_max, C), dtype=torch.uint8, device="cuda")
    dseg = torch.from_numpy(segs).to("cuda") if seg is not None else None
    N.mxfp8_quantize(_dev(v), rows, C, 1, dseg, nseg, q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp8_quantize_cols_segmented(v, segs)
    np.testing.assert_array_equal(s.cpu().numpy()[:rs.shape[0]], rs)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
