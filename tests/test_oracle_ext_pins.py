"""Pins for the oracle's two-sided window and additive bias (fwd_ex / bwd_ex).

The window [p - wl, p + wr] is checked against visible-key sets written out by
hand from each page's own window formula (tests/golden/visibility_ext.json)
and against the oracle's (causal, window) path, bit for bit, where the two
coincide.  The additive bias (ferrotensor's [batch, heads, seq_q, seq_k] mask,
size-1 dimensions broadcast) is checked against closed forms (zero bias, a
per-row constant, -inf entries as a key mask) and an independent torch fp64
route with autograd."""
import json
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def page_window(page, causal, window):
    """(wl, wr) of each page's window rule (negative = unbounded)."""
    if window <= 0:
        return -1, (0 if causal else -1)
    if page == "ferrotensor":
        return window - 1, (0 if causal else window - 1)
    if page == "brotensor":
        return (window - 1, 0) if causal else (window // 2, window // 2)
    if page == "forge":
        return window - 1, (0 if causal else -1)
    raise ValueError(page)


def test_golden_visible_sets_ext(oracle):
    cases = json.load(open(os.path.join(HERE, "golden", "visibility_ext.json")))["cases"]
    for c in cases:
        Tk, p, hd = c["Tk"], c["p"], 4
        wl, wr = page_window(c["page"], c["causal"], c["window"])
        P = oracle.probs_ex(np.zeros((1, 1, hd)), rnd((1, Tk, hd), 3), rnd((1, Tk, hd), 4), 0, 0, H=1, Hkv=1,
                            scale=0.5, window_left=wl, window_right=wr, q_offset=p)
        got = [j for j in range(Tk) if P[0, j] != 0.0]
        assert got == c["visible"], c["source"]
        np.testing.assert_allclose(P[0, got], 1.0 / len(got), rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal,window,q_offset", [(True, 0, 0), (True, 3, 2), (False, 3, 1), (False, 0, 0)])
def test_two_sided_window_equals_the_causal_window_path(oracle, causal, window, q_offset):
    q, k, v, do = rnd((2, 9, 16), 1), rnd((2, 9 + q_offset, 8), 2), rnd((2, 9 + q_offset, 8), 3), rnd((2, 9, 16), 4)
    wl, wr = page_window("ferrotensor", causal, window)
    kw = dict(H=2, Hkv=1, scale=0.4, softcap=1.7, q_offset=q_offset)
    o1, l1 = oracle.fwd(q, k, v, causal=causal, window=window, **kw)
    o2, l2 = oracle.fwd_ex(q, k, v, window_left=wl, window_right=wr, **kw)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    g1 = oracle.bwd(q, k, v, do, causal=causal, window=window, **kw)
    g2 = oracle.bwd_ex(q, k, v, do, window_left=wl, window_right=wr, **kw)
    for a, b in zip(g1, g2):
        assert np.array_equal(a, b)


def test_zero_bias_is_no_bias(oracle):
    q, k, v, do = rnd((2, 7, 8), 5), rnd((2, 7, 8), 6), rnd((2, 7, 8), 7), rnd((2, 7, 8), 8)
    kw = dict(H=2, Hkv=2, scale=0.5, window_left=3, window_right=1)
    o1, l1 = oracle.fwd_ex(q, k, v, **kw)
    o2, l2 = oracle.fwd_ex(q, k, v, bias=np.zeros((1, 1, 1, 1)), **kw)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_row_constant_bias_shifts_lse_only(oracle):
    """softmax(s + c_i) = softmax(s): O is unchanged and LSE moves by c_i."""
    B, T, H = 2, 6, 2
    q, k, v = rnd((B, T, H * 4), 9), rnd((B, T, 4), 10), rnd((B, T, 4), 11)
    c = rnd((B, H, T, 1), 12)
    kw = dict(H=H, Hkv=1, scale=0.6, window_right=0)
    o1, l1 = oracle.fwd_ex(q, k, v, **kw)
    o2, l2 = oracle.fwd_ex(q, k, v, bias=c, **kw)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(l2, l1 + c[..., 0], atol=1e-13)


def test_minus_inf_bias_is_a_key_mask(oracle):
    B, T = 2, 8
    q, k, v = rnd((B, T, 8), 13), rnd((B, T, 8), 14), rnd((B, T, 8), 15)
    m = (np.random.default_rng(16).random((B, T)) > 0.4).astype(np.float64)
    m[:, 0] = 1.0
    bias = np.where(m > 0.5, 0.0, -np.inf)[:, None, None, :]
    kw = dict(H=1, Hkv=1, scale=0.5, window_left=-1, window_right=-1)
    o1, l1 = oracle.fwd_ex(q, k, v, key_mask=m, **kw)
    o2, l2 = oracle.fwd_ex(q, k, v, bias=bias, **kw)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def torch_ex(q, k, v, *, H, Hkv, scale, wl, wr, softcap, q_offset, bias):
    B, Tq, _ = q.shape
    Tk = k.shape[1]
    hd = q.shape[2] // H
    G = H // Hkv
    qh = q.view(B, Tq, H, hd).permute(0, 2, 1, 3)
    kh = k.view(B, Tk, Hkv, hd).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vh = v.view(B, Tk, Hkv, hd).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    s = scale * qh @ kh.transpose(-1, -2)
    if softcap > 0:
        s = softcap * torch.tanh(s / softcap)
    s = s + torch.as_tensor(bias)
    pos = torch.arange(Tq)[:, None] + q_offset
    j = torch.arange(Tk)[None, :]
    allow = torch.ones(Tq, Tk, dtype=torch.bool)
    if wl >= 0:
        allow &= j >= pos - wl
    if wr >= 0:
        allow &= j <= pos + wr
    s = s.masked_fill(~allow, float("-inf"))
    o = (torch.softmax(s, dim=-1) @ vh).permute(0, 2, 1, 3).reshape(B, Tq, H * hd)
    return o, torch.logsumexp(s, dim=-1)


@pytest.mark.parametrize("bshape", [(2, 4, 9, 9), (1, 4, 1, 9), (2, 1, 9, 9), (1, 1, 9, 1)])
@pytest.mark.parametrize("wl,wr,softcap", [(-1, -1, 0.0), (3, 2, 0.0), (4, -1, 2.0), (-1, 0, 1.5)])
def test_bias_matches_torch_fp64_with_autograd(oracle, bshape, wl, wr, softcap):
    B, T, H, Hkv, hd = 2, 9, 4, 2, 4
    q, k, v, do = rnd((B, T, H * hd), 21), rnd((B, T, Hkv * hd), 22), rnd((B, T, Hkv * hd), 23), rnd((B, T, H * hd), 24)
    bias = rnd(bshape, 25)
    kw = dict(H=H, Hkv=Hkv, scale=1 / math.sqrt(hd), softcap=softcap, q_offset=0)
    o, lse = oracle.fwd_ex(q, k, v, window_left=wl, window_right=wr, bias=bias, **kw)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to, tl = torch_ex(tq, tk, tv, wl=wl, wr=wr, bias=bias, **kw)
    np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, tl.detach().numpy(), atol=1e-12)
    (to * torch.tensor(do)).sum().backward()
    g = oracle.bwd_ex(q, k, v, do, window_left=wl, window_right=wr, bias=bias, **kw)
    for a, t in zip(g, (tq, tk, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), atol=1e-11)


@pytest.mark.parametrize("wl,wr,softcap,q_offset", [(2, 1, 0.0, 0), (-1, 0, 1.3, 2), (3, -1, 0.9, 1)])
def test_ex_gradients_match_finite_differences(oracle, wl, wr, softcap, q_offset):
    """Central differences (h = 1e-6) of sum(O * dO) through fwd_ex, with a
    broadcast bias holding a -inf entry, against bwd_ex."""
    B, Tq, H, Hkv, hd = 1, 5, 2, 1, 4
    Tk = Tq + q_offset
    q, k, v, do = rnd((B, Tq, H * hd), 31), rnd((B, Tk, Hkv * hd), 32), rnd((B, Tk, Hkv * hd), 33), rnd((B, Tq, H * hd), 34)
    bias = rnd((1, H, Tq, Tk), 35)
    bias[0, 1, 3, 0] = -np.inf
    kw = dict(H=H, Hkv=Hkv, scale=0.5, window_left=wl, window_right=wr, softcap=softcap, q_offset=q_offset, bias=bias)
    loss = lambda q_, k_, v_: float((oracle.fwd_ex(q_, k_, v_, **kw)[0] * do).sum())
    grads = oracle.bwd_ex(q, k, v, do, **kw)
    h = 1e-6
    for idx, x in enumerate((q, k, v)):
        num = np.zeros_like(x)
        for mi in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[mi] += h
            xm[mi] -= h
            ap, am = [q, k, v], [q, k, v]
            ap[idx], am[idx] = xp, xm
            num[mi] = (loss(*ap) - loss(*am)) / (2 * h)
        err = np.linalg.norm(num - grads[idx]) / max(np.linalg.norm(num), 1e-30)
        assert err <= 1e-6, (idx, err)
