"""Pins for the fp64 oracle: facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself -- a closed
form, an invariant the pages state, an independent torch fp64 route with
autograd, finite differences, or visible-key sets written out by hand from
the pages' formulas (tests/golden/visibility.json) -- chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def problem(B=2, Tq=9, Tk=9, H=4, Hkv=2, hd=8, seed=0, dscale=1.0):
    q = rnd((B, Tq, H * hd), seed) * dscale
    k = rnd((B, Tk, Hkv * hd), seed + 1) * dscale
    v = rnd((B, Tk, Hkv * hd), seed + 2)
    do = rnd((B, Tq, H * hd), seed + 3)
    return q, k, v, do


FLAG_SETS = [
    dict(causal=False, window=0, softcap=0.0, q_offset=0, mask=False),
    dict(causal=True, window=0, softcap=0.0, q_offset=0, mask=False),
    dict(causal=True, window=3, softcap=0.0, q_offset=0, mask=False),
    dict(causal=True, window=4, softcap=2.5, q_offset=2, mask=False),
    dict(causal=False, window=3, softcap=0.0, q_offset=1, mask=False),
    dict(causal=False, window=0, softcap=1.5, q_offset=0, mask=True),
    dict(causal=True, window=5, softcap=3.0, q_offset=3, mask=True),
]


def make_mask(B, Tk, seed):
    m = (np.random.default_rng(seed).random((B, Tk)) > 0.3).astype(np.float64)
    m[:, 0] = 1.0  # keep every row non-empty for the smooth checks
    return m


def kwargs_of(f, B, Tk, H, Hkv, hd, seed=7):
    kw = dict(H=H, Hkv=Hkv, scale=1.0 / math.sqrt(hd), causal=f["causal"], window=f["window"],
              softcap=f["softcap"], q_offset=f["q_offset"])
    kw["key_mask"] = make_mask(B, Tk, seed) if f["mask"] else None
    return kw


# ---------------------------------------------------------------- golden sets
def test_golden_visible_sets(oracle):
    """Zero queries give a uniform P over exactly the visible keys the pages define."""
    cases = json.load(open(os.path.join(HERE, "golden", "visibility.json")))["cases"]
    for c in cases:
        Tk, p = c["Tk"], c["p"]
        hd = 4
        q = np.zeros((1, 1, hd))
        k = rnd((1, Tk, hd), 3)
        v = rnd((1, Tk, hd), 4)
        mask = None if c["mask"] is None else np.array(c["mask"], np.float64)
        P = oracle.probs(q, k, v, 0, 0, H=1, Hkv=1, scale=0.5, causal=c["causal"],
                         window=c["window"], q_offset=p, key_mask=mask)
        got = [j for j in range(Tk) if P[0, j] != 0.0]
        assert got == c["visible"], c["source"]
        np.testing.assert_allclose(P[0, got], 1.0 / len(got), rtol=0, atol=1e-15)


# ------------------------------------------------------------ normalisation
@pytest.mark.parametrize("f", FLAG_SETS)
def test_rows_sum_to_one(oracle, f):
    B, T, H, Hkv, hd = 2, 11, 4, 2, 8
    q, k, v, _ = problem(B, T, T, H, Hkv, hd, seed=11)
    kw = kwargs_of(f, B, T, H, Hkv, hd)
    for b in range(B):
        for h in range(H):
            P = oracle.probs(q, k, v, b, h, **kw)
            s = P.sum(axis=1)
            nonempty = s > 0
            np.testing.assert_allclose(s[nonempty], 1.0, rtol=0, atol=1e-12)
            assert (P >= 0).all()


# ------------------------------------------------------------- closed forms
def test_single_key_returns_v0(oracle):
    """Tk = 1: O = V_0 and LSE = the (capped) score of that key."""
    hd = 16
    q, k, v, _ = problem(1, 5, 1, 2, 1, hd, seed=21)
    for cap in (0.0, 0.7):
        o, lse = oracle.fwd(q, k, v, H=2, Hkv=1, scale=0.25, softcap=cap)
        for h in range(2):
            for i in range(5):
                s = 0.25 * float(np.dot(q[0, i, h * hd:(h + 1) * hd], k[0, 0]))
                st = cap * math.tanh(s / cap) if cap > 0 else s
                assert lse[0, h, i] == pytest.approx(st, abs=1e-14)
                np.testing.assert_allclose(o[0, i, h * hd:(h + 1) * hd], v[0, 0], atol=1e-14)


def test_identical_keys_average_visible_v(oracle):
    """All keys equal: P is uniform over the visible keys, O their mean of V."""
    T, hd = 10, 8
    q = rnd((1, T, hd), 31)
    k = np.tile(rnd((1, 1, hd), 32), (1, T, 1))
    v = rnd((1, T, hd), 33)
    o, _ = oracle.fwd(q, k, v, H=1, Hkv=1, scale=0.3, causal=True, window=4)
    for i in range(T):
        lo = max(0, i - 3)
        np.testing.assert_allclose(o[0, i], v[0, lo:i + 1].mean(axis=0), atol=1e-13)


def test_causal_row0(oracle):
    q, k, v, _ = problem(1, 6, 6, 1, 1, 8, seed=41)
    o, lse = oracle.fwd(q, k, v, H=1, Hkv=1, scale=0.5, causal=True)
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-15)
    assert lse[0, 0, 0] == pytest.approx(0.5 * float(np.dot(q[0, 0], k[0, 0])), abs=1e-14)


def test_two_key_softcap_closed_form(oracle):
    """Two visible keys: P_0 = sigmoid(st_0 - st_1), st = c tanh(s/c); LSE = logaddexp."""
    hd = 4
    q, k, v, _ = problem(1, 1, 2, 1, 1, hd, seed=51, dscale=2.0)
    for cap in (0.0, 0.5, 3.0, 50.0):
        o, lse = oracle.fwd(q, k, v, H=1, Hkv=1, scale=0.9, softcap=cap)
        s = [0.9 * float(np.dot(q[0, 0], k[0, j])) for j in range(2)]
        st = [cap * math.tanh(x / cap) if cap > 0 else x for x in s]
        p0 = 1.0 / (1.0 + math.exp(st[1] - st[0]))
        np.testing.assert_allclose(o[0, 0], p0 * v[0, 0] + (1 - p0) * v[0, 1], atol=1e-14)
        m = max(st)
        assert lse[0, 0, 0] == pytest.approx(m + math.log(math.exp(st[0] - m) + math.exp(st[1] - m)),
                                             abs=1e-14)


# ------------------------------------------------------ page equivalences
def test_window_at_least_T_is_unbounded(oracle):
    q, k, v, _ = problem(2, 12, 12, 4, 2, 8, seed=61)
    base = dict(H=4, Hkv=2, scale=0.35, causal=True)
    o0, l0 = oracle.fwd(q, k, v, window=0, **base)
    for w in (12, 13, 100):
        o1, l1 = oracle.fwd(q, k, v, window=w, **base)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_softcap_zero_is_off_and_large_cap_approaches_off(oracle):
    q, k, v, _ = problem(1, 7, 7, 2, 2, 8, seed=71)
    base = dict(H=2, Hkv=2, scale=0.35, causal=True)
    o0, l0 = oracle.fwd(q, k, v, **base)
    o1, l1 = oracle.fwd(q, k, v, softcap=0.0, **base)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    o2, l2 = oracle.fwd(q, k, v, softcap=1e7, **base)
    np.testing.assert_allclose(o2, o0, atol=1e-10)
    np.testing.assert_allclose(l2, l0, atol=1e-10)
    # a small cap really changes the result (the cap is applied, not ignored)
    o3, _ = oracle.fwd(q, k, v, softcap=0.2, **base)
    assert np.abs(o3 - o0).max() > 1e-3


def test_gqa_equals_mha_with_repeated_kv(oracle):
    """Hkv < H equals MHA on K/V repeated per group (consecutive heads share a KV head)."""
    B, T, H, Hkv, hd = 2, 9, 6, 2, 8
    q, k, v, do = problem(B, T, T, H, Hkv, hd, seed=81)
    G = H // Hkv
    rep = lambda x: np.repeat(x.reshape(B, T, Hkv, hd), G, axis=2).reshape(B, T, H * hd)
    kw = dict(scale=0.3, causal=True, window=4, softcap=2.0)
    o_g, l_g = oracle.fwd(q, k, v, H=H, Hkv=Hkv, **kw)
    o_m, l_m = oracle.fwd(q, rep(k), rep(v), H=H, Hkv=H, **kw)
    np.testing.assert_array_equal(o_g, o_m)
    np.testing.assert_array_equal(l_g, l_m)
    dq_g, dk_g, dv_g = oracle.bwd(q, k, v, do, H=H, Hkv=Hkv, **kw)
    dq_m, dk_m, dv_m = oracle.bwd(q, rep(k), rep(v), do, H=H, Hkv=H, **kw)
    np.testing.assert_allclose(dq_g, dq_m, atol=1e-13)
    fold = lambda x: x.reshape(B, T, Hkv, G, hd).sum(axis=3).reshape(B, T, Hkv * hd)
    np.testing.assert_allclose(dk_g, fold(dk_m), atol=1e-13)
    np.testing.assert_allclose(dv_g, fold(dv_m), atol=1e-13)


def test_prefix_mask_equals_truncated_cache(oracle):
    """A mask of L ones then zeros equals a cache cut to L keys, bit for bit."""
    B, Tq, Tk, H, hd = 1, 5, 16, 2, 8
    q, k, v, _ = problem(B, Tq, Tk, H, H, hd, seed=91)
    for L in (1, 7, 16):
        mask = (np.arange(Tk) < L).astype(np.float64)
        o1, l1 = oracle.fwd(q, k, v, H=H, Hkv=H, scale=0.4, key_mask=mask)
        o2, l2 = oracle.fwd(q, k[:, :L], v[:, :L], H=H, Hkv=H, scale=0.4)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_mask_keeps_a_key_only_above_one_half(oracle):
    """A key is valid iff its mask entry is > 0.5 (brotensor ops/flash_attention.h,
    flash_attention_forward and _backward contracts): entries of exactly 0.5 drop the
    key like 0 does, entries just above keep it like 1 does, bit for bit."""
    B, Tq, Tk, H, hd = 2, 6, 10, 2, 8
    q, k, v, do = problem(B, Tq, Tk, H, H, hd, seed=95)
    soft = np.array([[0.5, 1.0, 0.5000001, 0.0, 0.75, 0.5, 2.0, 0.49, 1.0, 0.5]] * B)
    hard = (soft > 0.5).astype(np.float64)
    assert 0 < hard.sum() < soft.size
    kw = dict(H=H, Hkv=H, scale=0.4, causal=False)
    o1, l1 = oracle.fwd(q, k, v, key_mask=soft, **kw)
    o2, l2 = oracle.fwd(q, k, v, key_mask=hard, **kw)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    for g1, g2 in zip(oracle.bwd(q, k, v, do, key_mask=soft, **kw), oracle.bwd(q, k, v, do, key_mask=hard, **kw)):
        assert np.array_equal(g1, g2)


def test_decode_rows_equal_prefill_tail(oracle):
    """Lq rows at q_offset = Tk - Lq equal the last Lq rows of causal prefill."""
    B, T, H, Hkv, hd = 2, 13, 4, 2, 8
    q, k, v, _ = problem(B, T, T, H, Hkv, hd, seed=101)
    for w in (0, 5):
        o_full, l_full = oracle.fwd(q, k, v, H=H, Hkv=Hkv, scale=0.3, causal=True, window=w)
        for Lq in (1, 4):
            o_d, l_d = oracle.fwd(q[:, T - Lq:], k, v, H=H, Hkv=Hkv, scale=0.3, causal=True,
                                  window=w, q_offset=T - Lq)
            assert np.array_equal(o_d, o_full[:, T - Lq:])
            assert np.array_equal(l_d, l_full[:, :, T - Lq:])


def test_fully_masked_row_is_zero_with_neg_inf_lse(oracle):
    q, k, v, do = problem(1, 4, 4, 1, 1, 8, seed=111)
    mask = np.array([0.0, 0.0, 1.0, 1.0])
    o, lse = oracle.fwd(q, k, v, H=1, Hkv=1, scale=0.3, causal=True, key_mask=mask)
    assert (o[0, :2] == 0).all() and np.isneginf(lse[0, 0, :2]).all()
    assert np.isfinite(lse[0, 0, 2:]).all()
    dq, dk, dv = oracle.bwd(q, k, v, do, H=1, Hkv=1, scale=0.3, causal=True, key_mask=mask)
    assert (dq[0, :2] == 0).all()
    assert (dk[0, :2] == 0).all() and (dv[0, :2] == 0).all()


# ------------------------------------------------------- LSE, D identity
@pytest.mark.parametrize("f", FLAG_SETS)
def test_lse_is_logsumexp_of_visible_scores(oracle, f):
    from scipy.special import logsumexp

    B, T, H, Hkv, hd = 2, 10, 4, 2, 8
    q, k, v, _ = problem(B, T, T, H, Hkv, hd, seed=121)
    kw = kwargs_of(f, B, T, H, Hkv, hd)
    _, lse = oracle.fwd(q, k, v, **kw)
    G = H // Hkv
    for b in range(B):
        for h in range(H):
            P = oracle.probs(q, k, v, b, h, **kw)
            qh = q[b, :, h * hd:(h + 1) * hd]
            kh = k[b, :, (h // G) * hd:(h // G + 1) * hd]
            s = kw["scale"] * qh @ kh.T
            if kw["softcap"] > 0:
                s = kw["softcap"] * np.tanh(s / kw["softcap"])
            for i in range(T):
                vis = P[i] > 0
                assert lse[b, h, i] == pytest.approx(logsumexp(s[i][vis]), abs=1e-12)


@pytest.mark.parametrize("f", FLAG_SETS)
def test_d_identity(oracle, f):
    """dO_i . O_i = sum_j P_ij (dO_i . V_j)."""
    B, T, H, Hkv, hd = 1, 9, 2, 1, 8
    q, k, v, do = problem(B, T, T, H, Hkv, hd, seed=131)
    kw = kwargs_of(f, B, T, H, Hkv, hd)
    o, _ = oracle.fwd(q, k, v, **kw)
    for h in range(H):
        P = oracle.probs(q, k, v, 0, h, **kw)
        doh = do[0, :, h * hd:(h + 1) * hd]
        lhs = (doh * o[0, :, h * hd:(h + 1) * hd]).sum(axis=1)
        rhs = (P * (doh @ v[0, :, :hd].T)).sum(axis=1)
        np.testing.assert_allclose(lhs, rhs, atol=1e-12)


# ------------------------------------------ independent torch fp64 route
def torch_attention(q, k, v, *, H, Hkv, scale, causal, window, softcap, q_offset, key_mask):
    """Textbook attention with an explicit boolean mask and torch.softmax (fp64)."""
    B, Tq, _ = q.shape
    Tk = k.shape[1]
    hd = q.shape[2] // H
    G = H // Hkv
    qh = q.view(B, Tq, H, hd).permute(0, 2, 1, 3)
    kh = k.view(B, Tk, Hkv, hd).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vh = v.view(B, Tk, Hkv, hd).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    s = scale * torch.matmul(qh, kh.transpose(-1, -2))
    if softcap > 0:
        s = softcap * torch.tanh(s / softcap)
    pos = torch.arange(Tq)[:, None] + q_offset
    j = torch.arange(Tk)[None, :]
    allow = torch.ones(Tq, Tk, dtype=torch.bool)
    if causal:
        allow &= j <= pos
    if window > 0:
        allow &= (pos - j).abs() < window
    allow = allow[None, None].expand(B, H, Tq, Tk)
    if key_mask is not None:
        km = torch.as_tensor(key_mask)
        km = km[None].expand(B, Tk) if km.dim() == 1 else km
        allow = allow & (km > 0.5)[:, None, None, :]
    s = s.masked_fill(~allow, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    p = torch.softmax(s, dim=-1)
    o = torch.matmul(p, vh).permute(0, 2, 1, 3).reshape(B, Tq, H * hd)
    return o, lse


@pytest.mark.parametrize("f", FLAG_SETS)
def test_matches_torch_fp64_forward_and_autograd(oracle, f):
    B, Tq, Tk, H, Hkv, hd = 2, 13, 13, 4, 2, 8
    if f["q_offset"]:
        Tk = Tq + f["q_offset"]
    q, k, v, do = problem(B, Tq, Tk, H, Hkv, hd, seed=141)
    kw = kwargs_of(f, B, Tk, H, Hkv, hd)
    o, lse = oracle.fwd(q, k, v, **kw)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    to, tl = torch_attention(tq, tk, tv, **kw)
    np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, tl.detach().numpy(), atol=1e-12)
    (to * torch.tensor(do)).sum().backward()
    dq, dk, dv = oracle.bwd(q, k, v, do, **kw)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


# ---------------------------------------------------- finite differences
@pytest.mark.parametrize("causal,window,softcap,mask,q_offset",
                         list(itertools.product([False, True], [0, 3], [0.0, 1.3], [False, True], [0]))
                         + [(True, 2, 0.9, True, 2)])
def test_finite_difference_gradients(oracle, causal, window, softcap, mask, q_offset):
    """Central differences (h = 1e-6) of L = sum(O * dO) on B=1, T<=8, H=2, Hkv=1, hd=4."""
    B, Tq, H, Hkv, hd = 1, 6, 2, 1, 4
    Tk = Tq + q_offset
    q, k, v, do = problem(B, Tq, Tk, H, Hkv, hd, seed=151, dscale=1.5)
    kw = dict(H=H, Hkv=Hkv, scale=0.5, causal=causal, window=window, softcap=softcap,
              q_offset=q_offset, key_mask=make_mask(B, Tk, 5) if mask else None)
    loss = lambda q_, k_, v_: float((oracle.fwd(q_, k_, v_, **kw)[0] * do).sum())
    grads = oracle.bwd(q, k, v, do, **kw)
    h = 1e-6
    for idx, x in enumerate((q, k, v)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            xp = x.copy(); xp[mi] += h
            xm = x.copy(); xm[mi] -= h
            args_p = [q, k, v]; args_p[idx] = xp
            args_m = [q, k, v]; args_m[idx] = xm
            num[mi] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.linalg.norm(num - grads[idx]) / max(np.linalg.norm(num), 1e-30)
        assert err <= 1e-6, (idx, err)
