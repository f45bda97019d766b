"""Two-sided windows and the additive score bias on the GPU against the fp64
oracle (fwd_ex / bwd_ex): every page's window rule, broadcast bias shapes,
-inf bias entries (a fully dropped row included), a bias together with a softcap
(the cap first, then the bias), and the plain causal/window calls reproduced bit
for bit.
Every call goes through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_attn_fwd_08_gb300 as A
from attention_attn_fwd_08_gb300 import synth
from helpers import compare_grads, compare_o_lse, f64, inputs

pytestmark = pytest.mark.gpu


def bias_of(shape, seed, holes=False):
    g = torch.Generator().manual_seed(seed)
    b = torch.randn(shape, generator=g, dtype=torch.float32) * 0.7
    if holes:
        b = b.masked_fill(torch.rand(shape, generator=g) < 0.2, float("-inf"))
    return b


def run_ex(dt, B, Tq, Tk, H, Hkv, hd, seed, wl=-1, wr=-1, softcap=0.0, q_offset=0, bias=None, backward=True):
    q, k, v, do = inputs(dt, B, Tq, Tk, H, Hkv, hd, seed, backward)
    kw = dict(H=H, Hkv=Hkv, scale=1.0 / math.sqrt(hd), window_left=wl, window_right=wr, softcap=softcap,
              q_offset=q_offset)
    bd = bias.cuda() if bias is not None else None
    o, lse = A.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), bias=bd, **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, hex(word)
    bnp = None if bias is None else bias.numpy().astype(np.float64)
    o_ref, lse_ref = oracle.fwd_ex(f64(q), f64(k), f64(v), bias=bnp, **kw)
    what = "%s B%d Tq%d Tk%d H%d/%d hd%d wl%d wr%d cap%g off%d bias=%s" % (
        dt, B, Tq, Tk, H, Hkv, hd, wl, wr, softcap, q_offset, None if bias is None else tuple(bias.shape))
    compare_o_lse(o, lse, o_ref, lse_ref, dt, what)
    if backward:
        g = A.attn_bwd_ex(q.cuda(), k.cuda(), v.cuda(), o, do.cuda(), lse, bias=bd, **kw)
        torch.cuda.synchronize()
        st, word = A.attn_get_device_status()
        assert st == A.OK, hex(word)
        compare_grads(g, oracle.bwd_ex(f64(q), f64(k), f64(v), f64(do), bias=bnp, **kw), dt, what)


# (wl, wr): brotensor's bidirectional window 100, forge's one-sided window 100,
# keys up to 30 ahead only, a causal window of 65, both sides unbounded
WINDOWS = [(50, 50), (99, -1), (-1, 30), (64, 0), (-1, -1)]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("wl,wr", WINDOWS)
def test_two_sided_windows(dt, hd, wl, wr):
    run_ex(dt, 2, 300, 300, 4, 2, hd, seed=800 + hd, wl=wl, wr=wr, softcap=20.0 if wr == -1 else 0.0)


@pytest.mark.parametrize("hd", [32, 96])
def test_two_sided_windows_padded_heads(hd):
    """hd 32 / 96 take the padded tensor-core kernels with a two-sided window; with a
    bias they take the CUDA-core kernels."""
    run_ex("bf16", 2, 300, 300, 4, 2, hd, seed=805 + hd, wl=50, wr=30)
    run_ex("f16", 1, 200, 230, 4, 2, hd, seed=806 + hd, wl=-1, wr=20, bias=bias_of((1, 4, 200, 230), 807))


def test_two_sided_window_with_q_offset_fp32():
    run_ex("f32", 1, 150, 190, 2, 1, 64, seed=810, wl=40, wr=10, q_offset=40)


@pytest.mark.parametrize("shape", [(2, 4, 260, 300), (1, 4, 1, 300), (2, 1, 260, 300), (1, 1, 260, 1)],
                         ids=["full", "per-head-key", "per-batch", "per-query-row"])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_additive_bias(dt, shape):
    run_ex(dt, 2, 260, 300, 4, 2, 128, seed=820, wl=-1, wr=40, bias=bias_of(shape, 821))


@pytest.mark.parametrize("hd", [64, 128])
def test_bias_with_minus_inf_entries(hd):
    """-inf drops pairs; row 5 of every head drops every key (O = 0, LSE = -inf)."""
    b = bias_of((2, 4, 200, 200), 830, holes=True)
    b[:, :, 5, :] = float("-inf")
    run_ex("bf16", 2, 200, 200, 4, 2, hd, seed=831, wl=-1, wr=0, bias=b)


@pytest.mark.parametrize("dt,hd,softcap", [("bf16", 128, 5.0), ("f16", 64, 30.0), ("bf16", 128, 50.0)])
def test_bias_with_softcap(dt, hd, softcap):
    """The tensor-core kernels with the cap applied before the bias: a small softcap
    (scores beyond the fitted polynomial's range: the exp-based tanh), moderate ones
    (the polynomial tiers), several tiles, a ragged tail and -inf bias entries."""
    b = bias_of((2, 4, 300, 300), 841, holes=True)
    run_ex(dt, 2, 300, 300, 4, 2, hd, seed=840, wl=30, wr=30, softcap=softcap, bias=b)
    run_ex(dt, 1, 260, 260, 4, 2, hd, seed=842, wl=-1, wr=0, softcap=softcap, bias=bias_of((1, 4, 260, 260), 843))


def test_bias_with_softcap_padded_head_takes_the_cuda_core_kernels():
    run_ex("bf16", 1, 140, 140, 2, 1, 96, seed=844, wl=30, wr=30, softcap=5.0, bias=bias_of((1, 2, 140, 140), 845))


def test_bias_fp32():
    run_ex("f32", 1, 100, 120, 2, 2, 64, seed=850, wl=-1, wr=-1, bias=bias_of((1, 2, 100, 120), 851))


@pytest.mark.parametrize("causal,window", [(True, 0), (True, 77), (False, 77), (False, 0)])
def test_ex_reproduces_causal_window_calls_bit_for_bit(causal, window):
    q, k, v, do = (t.cuda() for t in inputs("bf16", 2, 333, 333, 8, 2, 128, 860, True))
    wl = window - 1 if window > 0 else -1
    wr = 0 if causal else (window - 1 if window > 0 else -1)
    kw = dict(H=8, Hkv=2, softcap=0.0)
    o1, l1 = A.attn_fwd(q, k, v, causal=causal, window=window, **kw)
    o2, l2 = A.attn_fwd_ex(q, k, v, window_left=wl, window_right=wr, **kw)
    g1 = A.attn_bwd(q, k, v, o1, do, l1, causal=causal, window=window, **kw)
    g2 = A.attn_bwd_ex(q, k, v, o2, do, l2, window_left=wl, window_right=wr, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
