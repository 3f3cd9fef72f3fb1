"""Failure detection on the device, in forms that cannot fault the GPU.

1. A bounded wait that runs out. moe_selftest_wait_timeout makes one warp wait
   on an mbarrier that nothing arrives on (limit ~1 ms) while a second warp
   waits with the GEMMs' own ~2 s limit; the expired wait must set
   MOE_ERR_TIMEOUT in the device error word and stop the second warp through
   the block's abort flag. The context must stay usable: a whole layer runs
   after it and matches a run before it bit for bit.

2. Caller-supplied row indices out of range. moe_permute, moe_combine_fwd,
   moe_combine_bwd, moe_permute_bwd and the two MXFP8 dispatch calls take
   dest_row / topk_idx from the caller. One index is corrupted on the host to
   point at a guard row that the test allocates past the R routed rows (or a
   guard expert row of w_router), so even a kernel that missed the check would
   only touch memory the test owns. The kernel must skip that pair, set
   MOE_ERR_DEVICE_INDEX, leave the guard rows untouched, and compute every
   other pair exactly as before.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_prefix_gb300 import _native as N
from mixture_experts_layer_prefix_gb300 import build as B
from mixture_experts_layer_prefix_gb300 import layer as L
from mixture_experts_layer_prefix_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4            # guard rows past the R routed rows
SENTINEL = 12288.0   # 3 * 2^12, bf16-exact; marks guard rows that must stay untouched


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    N.load()
    assert N.moe_get_device_error() == 0


def _routing(T, k, E, seed):
    """A valid routing as moe_route lays it out: topk_idx, dest_row, offsets."""
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    counts = np.bincount(idx.ravel(), minlength=E)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    dest = np.empty((T, k), np.int32)
    fill = offs[:-1].copy()
    for t in range(T):
        for j in range(k):
            dest[t, j] = fill[idx[t, j]]
            fill[idx[t, j]] += 1
    return idx, dest, offs


def _bf16(rng, *shape):
    return torch.from_numpy(synth.round_bf16(rng.standard_normal(shape).astype(np.float32))).cuda().to(torch.bfloat16)


def _small_layer():
    s = synth.MoEShape("after_timeout", 300, 128, 8, 2, 128, "bf16", 0.02)
    inp = synth.Inputs(s, seed=4)
    p = L.params_from_inputs(inp, N.MOE_BF16)
    b = L.Buffers(s.T, s.d, s.E, s.k, s.f, N.MOE_BF16)
    L.forward(p, b)
    L.backward(p, b)
    torch.cuda.synchronize()
    return [t.clone() for t in (b.y, b.dx, b.dw_gate, b.dw_down, b.dw_router)]


def test_bounded_wait_times_out_and_the_context_survives():
    before = _small_layer()
    assert N.moe_get_device_error() == 0
    out = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    N.moe_selftest_wait_timeout(2_000_000, out)  # ~1 ms at 2 GHz
    assert N.moe_get_device_error() == 7          # MOE_ERR_TIMEOUT, read and cleared
    assert out[:2].tolist() == [0, 0]             # both waits gave up: one expired, one aborted
    assert N.moe_get_device_error() == 0          # the word was cleared
    after = _small_layer()
    assert N.moe_get_device_error() == 0
    for a, c in zip(before, after):
        assert torch.equal(a, c)


def test_selftest_rejects_bad_arguments():
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    for cycles in (0, -5, 5_000_000_000):
        with pytest.raises(N.MoEError):
            N.moe_selftest_wait_timeout(cycles, out)


T, D, K, E = 96, 256, 2, 6
R = T * K
BAD_T, BAD_J = 17, 1


def _case(seed=3):
    rng = np.random.default_rng(seed)
    idx, dest, offs = _routing(T, K, E, seed)
    bad = dest.copy()
    bad[BAD_T, BAD_J] = R  # the first guard row
    return rng, idx, dest, bad, offs


def _guarded(rows, d, dtype=torch.bfloat16, fill=SENTINEL):
    return torch.full((rows + GUARD, d), fill, dtype=dtype, device="cuda")


def test_permute_skips_a_row_index_past_R():
    rng, idx, dest, bad, offs = _case()
    x = _bf16(rng, T, D)
    xp = _guarded(R, D)
    N.moe_permute(x, N.MOE_BF16, T, D, K, torch.from_numpy(bad).cuda(), xp)
    assert N.moe_get_device_error() == 6  # MOE_ERR_DEVICE_INDEX
    assert torch.all(xp[R:] == SENTINEL)
    xn = x.float().cpu().numpy()
    got = xp.float().cpu().numpy()
    for t in range(T):
        for j in range(K):
            if (t, j) != (BAD_T, BAD_J):
                np.testing.assert_array_equal(got[dest[t, j]], xn[t])
    assert np.all(got[dest[BAD_T, BAD_J]] == SENTINEL)  # the row nobody wrote


def test_combine_fwd_skips_a_row_index_past_R():
    rng, idx, dest, bad, offs = _case()
    yp = _bf16(rng, R + GUARD, D)
    g = torch.from_numpy(rng.random((T, K)).astype(np.float32)).cuda()
    y_ok = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    y_bad = torch.empty_like(y_ok)
    N.moe_combine_fwd(yp, g, torch.from_numpy(dest).cuda(), N.MOE_BF16, T, D, K, y_ok)
    assert N.moe_get_device_error() == 0
    # the corrupted pair contributes nothing: same as a zero gate on it
    g0 = g.clone()
    g0[BAD_T, BAD_J] = 0.0
    y_zero = torch.empty_like(y_ok)
    N.moe_combine_fwd(yp, g0, torch.from_numpy(dest).cuda(), N.MOE_BF16, T, D, K, y_zero)
    N.moe_combine_fwd(yp, g, torch.from_numpy(bad).cuda(), N.MOE_BF16, T, D, K, y_bad)
    assert N.moe_get_device_error() == 6
    assert torch.equal(y_bad, y_zero)
    rows = [t for t in range(T) if t != BAD_T]
    assert torch.equal(y_bad[rows], y_ok[rows])


def test_combine_bwd_skips_a_row_index_past_R():
    rng, idx, dest, bad, offs = _case()
    dy = _bf16(rng, T, D)
    yp = _bf16(rng, R + GUARD, D)
    g = torch.from_numpy(rng.random((T, K)).astype(np.float32)).cuda()
    dyp_ok = _guarded(R, D)
    dg_ok = torch.empty((T, K), dtype=torch.float32, device="cuda")
    N.moe_combine_bwd(dy, yp, g, torch.from_numpy(dest).cuda(), N.MOE_BF16, T, D, K, dyp_ok, dg_ok)
    assert N.moe_get_device_error() == 0
    dyp = _guarded(R, D)
    dg = torch.empty_like(dg_ok)
    N.moe_combine_bwd(dy, yp, g, torch.from_numpy(bad).cuda(), N.MOE_BF16, T, D, K, dyp, dg)
    assert N.moe_get_device_error() == 6
    assert torch.all(dyp[R:] == SENTINEL)
    assert float(dg[BAD_T, BAD_J]) == 0.0
    keep = np.ones((T, K), bool)
    keep[BAD_T, BAD_J] = False
    kt = torch.from_numpy(keep).cuda()
    assert torch.equal(dg[kt], dg_ok[kt])
    rows = torch.from_numpy(dest[keep]).long().cuda()
    assert torch.equal(dyp[rows], dyp_ok[rows])


def test_permute_bwd_skips_bad_rows_and_bad_experts():
    rng, idx, dest, bad, offs = _case()
    dxp = _bf16(rng, R + GUARD, D)
    dl = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
    wr = _bf16(rng, E + 1, D)  # row E is a guard expert row
    dx_ok = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    idx_d = torch.from_numpy(idx).cuda()
    N.moe_permute_bwd(dxp, N.MOE_BF16, T, D, E, K, torch.from_numpy(dest).cuda(), idx_d, dl, wr, dx_ok)
    assert N.moe_get_device_error() == 0
    # a bad row index: that pair (its dx_perm row and its router term) is skipped
    dx = torch.empty_like(dx_ok)
    N.moe_permute_bwd(dxp, N.MOE_BF16, T, D, E, K, torch.from_numpy(bad).cuda(), idx_d, dl, wr, dx)
    assert N.moe_get_device_error() == 6
    rows = [t for t in range(T) if t != BAD_T]
    assert torch.equal(dx[rows], dx_ok[rows])
    # a bad expert index (E: the guard row of w_router) on another token
    bad_e = idx.copy()
    bad_e[BAD_T + 1, 0] = E
    dx2 = torch.empty_like(dx_ok)
    N.moe_permute_bwd(dxp, N.MOE_BF16, T, D, E, K, torch.from_numpy(dest).cuda(), torch.from_numpy(bad_e).cuda(),
                      dl, wr, dx2)
    assert N.moe_get_device_error() == 6
    rows = [t for t in range(T) if t != BAD_T + 1]
    assert torch.equal(dx2[rows], dx_ok[rows])
    # that token keeps only its other pair (expert-path row and router term)
    want = dxp[dest[BAD_T + 1, 1]].float() + dl[BAD_T + 1, idx[BAD_T + 1, 1]] * wr[idx[BAD_T + 1, 1]].float()
    np.testing.assert_allclose(dx2[BAD_T + 1].float().cpu().numpy(), want.cpu().numpy(), rtol=1e-2, atol=1e-2)


def test_mxfp8_dispatch_and_combine_bwd_skip_bad_rows():
    rng, idx, dest, bad, offs = _case()
    x = _bf16(rng, T, D)
    dy = _bf16(rng, T, D)
    yp = _bf16(rng, R + GUARD, D)
    g = torch.from_numpy(rng.random((T, K)).astype(np.float32)).cuda()
    nsc = N.moe_mxfp8_row_scales_size(R, E, D)
    slack = 4 * nsc + (1 << 16)  # scale chunks a missed check could reach stay inside this buffer
    idx_d, offs_d = torch.from_numpy(idx).cuda(), torch.from_numpy(offs).cuda()

    def dispatch(dr):
        q = torch.zeros((R + GUARD, D), dtype=torch.uint8, device="cuda")
        sc = torch.zeros(slack, dtype=torch.uint8, device="cuda")
        xp = _guarded(R, D)
        N.moe_permute_mxfp8(x, T, D, K, E, torch.from_numpy(dr).cuda(), idx_d, offs_d, q, sc, xp)
        return q, sc, xp

    q0, sc0, xp0 = dispatch(dest)
    assert N.moe_get_device_error() == 0
    q1, sc1, xp1 = dispatch(bad)
    assert N.moe_get_device_error() == 6
    assert torch.all(q1[R:] == 0) and torch.all(xp1[R:] == SENTINEL) and torch.all(sc1[nsc:] == 0)
    keep = np.ones((T, K), bool)
    keep[BAD_T, BAD_J] = False
    rows = torch.from_numpy(dest[keep]).long().cuda()
    assert torch.equal(q1[rows], q0[rows]) and torch.equal(xp1[rows], xp0[rows])

    # an expert index that does not own the pair's row is refused too
    wrong_e = idx.copy()
    wrong_e[BAD_T, BAD_J] = (idx[BAD_T, BAD_J] + 1) % E
    q2 = torch.zeros((R + GUARD, D), dtype=torch.uint8, device="cuda")
    sc2 = torch.zeros(slack, dtype=torch.uint8, device="cuda")
    N.moe_permute_mxfp8(x, T, D, K, E, torch.from_numpy(dest).cuda(), torch.from_numpy(wrong_e).cuda(), offs_d, q2,
                        sc2, None)
    assert N.moe_get_device_error() == 6
    assert torch.equal(q2[rows], q0[rows])

    def cbwd(dr):
        q = torch.zeros((R + GUARD, D), dtype=torch.uint8, device="cuda")
        sc = torch.zeros(slack, dtype=torch.uint8, device="cuda")
        dyp = _guarded(R, D)
        dg = torch.empty((T, K), dtype=torch.float32, device="cuda")
        N.moe_combine_bwd_mxfp8(dy, yp, g, torch.from_numpy(dr).cuda(), idx_d, offs_d, T, D, K, E, q, sc, dyp, dg)
        return q, sc, dyp, dg

    c0 = cbwd(dest)
    assert N.moe_get_device_error() == 0
    c1 = cbwd(bad)
    assert N.moe_get_device_error() == 6
    assert torch.all(c1[0][R:] == 0) and torch.all(c1[2][R:] == SENTINEL) and torch.all(c1[1][nsc:] == 0)
    assert torch.equal(c1[0][rows], c0[0][rows]) and torch.equal(c1[2][rows], c0[2][rows])
    assert float(c1[3][BAD_T, BAD_J]) == 0.0
