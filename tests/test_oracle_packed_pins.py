"""Pins of the packed fused-QKV oracle (oracle.packed_qkv_fwd / packed_qkv_bwd, a row
by row numpy restatement of brotensor ops/flash_attention.h,
flash_attention_packed_qkv_forward / _backward) against things other than itself:
the C oracle run on each sequence as its own batch with the two-sided window
(|r - j| <= window/2 is window_left = window_right = window // 2), the closed form
of one-row sequences, and finite differences of the forward."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def packing(lengths):
    L = int(sum(lengths))
    sb = np.zeros((L, 2), np.int32)
    s = 0
    for n in lengths:
        sb[s:s + n] = (s, s + n)
        s += n
    return sb


def split(qkv, H):
    L, C = qkv.shape
    hd = C // (3 * H)
    return qkv[:, :H * hd], qkv[:, H * hd:2 * H * hd], qkv[:, 2 * H * hd:], hd


@pytest.mark.parametrize("window", [0, 1, 5, 8])
def test_packed_matches_per_sequence_c_oracle(window):
    rng = np.random.default_rng(7 + window)
    lengths, H, scale = [9, 1, 23, 4, 17], 3, 0.31
    sb = packing(lengths)
    L = len(sb)
    qkv = rng.standard_normal((L, 3 * H * 8))
    do = rng.standard_normal((L, H * 8))
    o, lse = oracle.packed_qkv_fwd(qkv, sb, H=H, scale=scale, window=window)
    dqkv = oracle.packed_qkv_bwd(qkv, do, sb, H=H, scale=scale, window=window)
    q, k, v, hd = split(qkv, H)
    w = window // 2 if window > 0 else -1
    s = 0
    for n in lengths:
        kw = dict(H=H, Hkv=H, scale=scale, window_left=w, window_right=w)
        o2, l2 = oracle.fwd_ex(q[None, s:s + n], k[None, s:s + n], v[None, s:s + n], **kw)
        np.testing.assert_allclose(o[s:s + n], o2[0], atol=1e-12)
        np.testing.assert_allclose(lse[:, s:s + n], l2[0], atol=1e-12)
        gq, gk, gv = oracle.bwd_ex(q[None, s:s + n], k[None, s:s + n], v[None, s:s + n], do[None, s:s + n], **kw)
        np.testing.assert_allclose(dqkv[s:s + n], np.concatenate([gq[0], gk[0], gv[0]], axis=1), atol=1e-12)
        s += n


def test_one_row_sequences_closed_form():
    """A row that is its own sequence sees only itself: O = v_r, LSE = scale q_r.k_r,
    and every gradient but dV = dO is zero (P = 1, dS = 0)."""
    rng = np.random.default_rng(3)
    H, hd, L = 2, 4, 6
    sb = packing([1] * L)
    qkv = rng.standard_normal((L, 3 * H * hd))
    do = rng.standard_normal((L, H * hd))
    q, k, v, _ = split(qkv, H)
    o, lse = oracle.packed_qkv_fwd(qkv, sb, H=H, scale=0.5)
    np.testing.assert_allclose(o, v, atol=1e-14)
    ref = 0.5 * (q.reshape(L, H, hd) * k.reshape(L, H, hd)).sum(-1).T
    np.testing.assert_allclose(lse, ref, atol=1e-14)
    d = oracle.packed_qkv_bwd(qkv, do, sb, H=H, scale=0.5)
    np.testing.assert_allclose(d[:, :2 * H * hd], 0.0, atol=1e-14)
    np.testing.assert_allclose(d[:, 2 * H * hd:], do, atol=1e-14)


def test_packed_bwd_finite_differences():
    rng = np.random.default_rng(11)
    H, hd = 2, 4
    sb = packing([3, 5])
    L = len(sb)
    qkv = rng.standard_normal((L, 3 * H * hd))
    do = rng.standard_normal((L, H * hd))
    f = lambda x: float((oracle.packed_qkv_fwd(x, sb, H=H, scale=0.4, window=4)[0] * do).sum())
    g = oracle.packed_qkv_bwd(qkv, do, sb, H=H, scale=0.4, window=4)
    eps = 1e-6
    for r, c in ((0, 0), (2, 9), (4, 17), (7, 23), (5, 3)):
        x1, x2 = qkv.copy(), qkv.copy()
        x1[r, c] += eps
        x2[r, c] -= eps
        assert abs((f(x1) - f(x2)) / (2 * eps) - g[r, c]) < 1e-6
