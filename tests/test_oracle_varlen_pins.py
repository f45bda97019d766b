"""Pins for the oracle's packed variable-length attention (brotensor
ops/flash_attention.h, flash_attention_varlen_forward / _backward).

The oracle runs each sequence as its own batch of one.  These tests check it
against routes that share none of that: a torch fp64 attention over the whole
packed tensor with an explicit block-diagonal mask and autograd, the dense
batched oracle when every sequence has the same length, and the independence
of sequences (changing one changes no other)."""
import math

import numpy as np
import pytest
import torch


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def packed(cu_q, cu_k, H, Hkv, hd, seed):
    tq, tk = int(cu_q[-1]) + 3, int(cu_k[-1]) + 2  # a few rows outside every sequence
    return (rnd((tq, H * hd), seed), rnd((tk, Hkv * hd), seed + 1), rnd((tk, Hkv * hd), seed + 2),
            rnd((tq, H * hd), seed + 3))


def torch_packed(q, k, v, cu_q, cu_k, *, H, Hkv, scale, causal, window, softcap):
    """Whole packed tensors, one explicit [total_q, total_k] mask: same sequence,
    positions counted from each sequence's first row (fp64, torch.softmax)."""
    tq, tk = q.shape[0], k.shape[0]
    hd = q.shape[1] // H
    G = H // Hkv
    seq_q = torch.full((tq,), -1, dtype=torch.long)
    seq_k = torch.full((tk,), -2, dtype=torch.long)
    pos_q = torch.zeros(tq, dtype=torch.long)
    pos_k = torch.zeros(tk, dtype=torch.long)
    for b in range(len(cu_q) - 1):
        seq_q[cu_q[b]:cu_q[b + 1]] = b
        seq_k[cu_k[b]:cu_k[b + 1]] = b
        pos_q[cu_q[b]:cu_q[b + 1]] = torch.arange(cu_q[b + 1] - cu_q[b])
        pos_k[cu_k[b]:cu_k[b + 1]] = torch.arange(cu_k[b + 1] - cu_k[b])
    allow = seq_q[:, None] == seq_k[None, :]
    if causal:
        allow &= pos_k[None, :] <= pos_q[:, None]
    if window > 0:
        allow &= (pos_q[:, None] - pos_k[None, :]).abs() < window
    qh = q.view(tq, H, hd).permute(1, 0, 2)
    kh = k.view(tk, Hkv, hd).permute(1, 0, 2).repeat_interleave(G, dim=0)
    vh = v.view(tk, Hkv, hd).permute(1, 0, 2).repeat_interleave(G, dim=0)
    s = scale * qh @ kh.transpose(1, 2)
    if softcap > 0:
        s = softcap * torch.tanh(s / softcap)
    s = s.masked_fill(~allow[None], float("-inf"))
    lse = torch.logsumexp(s, dim=-1)                          # [H, tq]
    live = allow.any(dim=1)                                   # rows that see a key
    p = torch.softmax(s.masked_fill(~live[None, :, None], 0.0), dim=-1) * live[None, :, None]
    o = (p @ vh).permute(1, 0, 2).reshape(tq, H * hd)
    return o, lse


CASES = [
    dict(causal=True, window=0, softcap=0.0),
    dict(causal=False, window=0, softcap=0.0),
    dict(causal=True, window=3, softcap=2.0),
    dict(causal=False, window=4, softcap=0.0),
]


@pytest.mark.parametrize("f", CASES, ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_varlen_matches_packed_torch_with_autograd(oracle, f):
    H, Hkv, hd = 4, 2, 8
    # ragged, an empty sequence, and (non-causal only) query and key lengths that differ
    cu_q = [0, 5, 5, 12, 21, 22]
    cu_k = [0, 5, 5, 12, 21, 22] if f["causal"] else [0, 7, 8, 12, 16, 26]
    q, k, v, do = packed(cu_q, cu_k, H, Hkv, hd, seed=11)
    kw = dict(H=H, Hkv=Hkv, scale=1.0 / math.sqrt(hd), **f)
    o, lses = oracle.varlen_fwd(q, k, v, cu_q, cu_k, **kw)
    tq_, tk_, tv_ = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to, tl = torch_packed(tq_, tk_, tv_, cu_q, cu_k, **kw)
    inside = np.zeros(q.shape[0], bool)
    inside[cu_q[0]:cu_q[-1]] = True
    np.testing.assert_allclose(o[inside], to.detach().numpy()[inside], atol=1e-12)
    assert not o[~inside].any()
    for b, lb in enumerate(lses):
        np.testing.assert_allclose(lb, tl.detach().numpy()[:, cu_q[b]:cu_q[b + 1]], atol=1e-12)
    (to * torch.tensor(do) * torch.tensor(inside[:, None], dtype=torch.float64)).sum().backward()
    dq, dk, dv = oracle.varlen_bwd(q, k, v, do, cu_q, cu_k, **kw)
    np.testing.assert_allclose(dq, tq_.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk_.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv_.grad.numpy(), atol=1e-11)


def test_varlen_sequence_without_keys(oracle):
    """A sequence with queries but no keys: O = 0, LSE = -inf, zero gradients."""
    H, Hkv, hd = 2, 1, 4
    cu_q, cu_k = [0, 3, 6], [0, 4, 4]
    q, k, v, do = packed(cu_q, cu_k, H, Hkv, hd, seed=3)
    kw = dict(H=H, Hkv=Hkv, scale=0.5, causal=False)
    o, lses = oracle.varlen_fwd(q, k, v, cu_q, cu_k, **kw)
    assert not o[3:6].any() and np.all(lses[1] == -np.inf)
    dq, dk, dv = oracle.varlen_bwd(q, k, v, do, cu_q, cu_k, **kw)
    assert not dq[3:6].any()


def test_equal_lengths_equal_the_dense_batch(oracle):
    B, T, H, Hkv, hd = 3, 7, 4, 2, 8
    cu = [0, 7, 14, 21]
    q, k, v, do = (x[:21] for x in packed(cu, cu, H, Hkv, hd, seed=5))
    kw = dict(H=H, Hkv=Hkv, scale=0.35, causal=True, window=5, softcap=3.0)
    o, lses = oracle.varlen_fwd(q, k, v, cu, cu, **kw)
    od, ld = oracle.fwd(q.reshape(B, T, -1), k.reshape(B, T, -1), v.reshape(B, T, -1), **kw)
    np.testing.assert_array_equal(o, od.reshape(B * T, -1))
    np.testing.assert_array_equal(np.stack(lses), ld)
    g = oracle.varlen_bwd(q, k, v, do, cu, cu, **kw)
    gd = oracle.bwd(q.reshape(B, T, -1), k.reshape(B, T, -1), v.reshape(B, T, -1), do.reshape(B, T, -1), **kw)
    for a, b in zip(g, gd):
        np.testing.assert_array_equal(a, b.reshape(a.shape))


def test_sequences_are_independent(oracle):
    H, Hkv, hd = 2, 2, 4
    cu = [0, 4, 9, 15]
    q, k, v, _ = packed(cu, cu, H, Hkv, hd, seed=9)
    kw = dict(H=H, Hkv=Hkv, scale=0.5, causal=True)
    o1, _ = oracle.varlen_fwd(q, k, v, cu, cu, **kw)
    k2, v2 = k.copy(), v.copy()
    k2[4:9] += 1.0
    v2[4:9] -= 2.0
    o2, _ = oracle.varlen_fwd(q, k2, v2, cu, cu, **kw)
    np.testing.assert_array_equal(o1[:4], o2[:4])
    np.testing.assert_array_equal(o1[9:], o2[9:])
    assert np.abs(o1[4:9] - o2[4:9]).max() > 0.1
