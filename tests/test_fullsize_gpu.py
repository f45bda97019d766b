"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (the same C-ABI calls on the same shapes).

The CUDA path runs on the whole problem; the oracle recomputes sampled
blocks.  A block is an exact sub-problem: attention is independent per
(batch, KV-head group), and a query row depends only on the keys it can see,
so slicing the query rows [r0, r1) with their visible keys [k0, k1) and
shifting q_offset by k0 leaves every sampled output unchanged.  dK/dV are
compared only on keys whose every viewing query lies inside the block.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_attn_fwd_08_gb300 as A
from attention_attn_fwd_08_gb300 import synth
from helpers import compare_grads, compare_o_lse, f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def heads(x, b, h0, h1, hd):
    return x[b:b + 1, :, h0 * hd:h1 * hd]


def sample_block(w, inp, gpu, b, kvh, r0, r1, k0, k1, grad_keys=None):
    """Compare O/LSE (and dQ, dK/dV on grad_keys) of rows [r0,r1) of group (b, kvh)."""
    G, hd = w.H // w.Hkv, w.hd
    h0, h1 = kvh * G, (kvh + 1) * G
    q = f64(heads(inp["q"], b, h0, h1, hd)[:, r0:r1])
    k = f64(heads(inp["k"], b, kvh, kvh + 1, hd)[:, k0:k1])
    v = f64(heads(inp["v"], b, kvh, kvh + 1, hd)[:, k0:k1])
    km = None
    if "key_mask" in inp:
        km = f64(inp["key_mask"][b, k0:k1])
    kw = dict(H=G, Hkv=1, scale=w.scale, causal=w.causal, window=w.window, softcap=w.softcap,
              q_offset=w.q_offset + r0 - k0, key_mask=km)
    o_ref, lse_ref = oracle.fwd(q, k, v, **kw)
    o_g = heads(gpu["o"], b, h0, h1, hd)[:, r0:r1]
    lse_g = gpu["lse"][b:b + 1, h0:h1, r0:r1]
    what = "%s b%d kvh%d rows[%d,%d)" % (w.name, b, kvh, r0, r1)
    compare_o_lse(o_g, lse_g, o_ref, lse_ref, w.dtype, what)
    if grad_keys is None:
        return
    do = f64(heads(inp["do"], b, h0, h1, hd)[:, r0:r1])
    dq, dk, dv = oracle.bwd(q, k, v, do, **kw)
    g0, g1 = grad_keys
    dq_g = heads(gpu["dq"], b, h0, h1, hd)[:, r0:r1]
    dk_g = heads(gpu["dk"], b, kvh, kvh + 1, hd)[:, g0:g1]
    dv_g = heads(gpu["dv"], b, kvh, kvh + 1, hd)[:, g0:g1]
    compare_grads((dq_g, dk_g, dv_g), (dq, dk[:, g0 - k0:g1 - k0], dv[:, g0 - k0:g1 - k0]), w.dtype, what)


def run_gpu(w, inp):
    dev = "cuda"
    qd, kd, vd = inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev)
    km = inp["key_mask"].to(dev) if "key_mask" in inp else None
    kw = dict(H=w.H, Hkv=w.Hkv, scale=w.scale, causal=w.causal, window=w.window, softcap=w.softcap,
              q_offset=w.q_offset, key_mask=km)
    out = {}
    if w.decode:
        o, lse = A.attn_decode(qd, kd, vd, **kw)
    else:
        o, lse = A.attn_fwd(qd, kd, vd, **kw)
    out["o"], out["lse"] = o, lse
    if w.backward:
        dq, dk, dv = A.attn_bwd(qd, kd, vd, o, inp["do"].to(dev), lse, **kw)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    return {k: v.cpu() for k, v in out.items()}


def test_gqa_prefill_fwd_bwd_full():
    w = synth.WORKLOADS["gqa_prefill"]
    inp = synth.make_inputs(w)
    gpu = run_gpu(w, inp)
    T = w.Tq
    # last 256 rows: every viewer of keys [T-256, T) is inside, so dK/dV there are exact
    sample_block(w, inp, gpu, 3, 5, T - 256, T, 0, T, grad_keys=(T - 256, T))
    sample_block(w, inp, gpu, 0, 0, T - 128, T, 0, T, grad_keys=(T - 128, T))
    sample_block(w, inp, gpu, 1, 2, 1000, 1100, 0, 1100)
    sample_block(w, inp, gpu, 2, 7, 0, 130, 0, 130)


def test_swa_softcap_fwd_bwd_full():
    w = synth.WORKLOADS["swa_softcap"]
    inp = synth.make_inputs(w)
    gpu = run_gpu(w, inp)
    W = w.window
    # keys [j0, j0+256) are seen by rows [j0, j0+256+W-1), which see keys [j0-W+1, ...)
    j0 = 4096
    sample_block(w, inp, gpu, 1, 2, j0, j0 + 256 + W - 1, j0 - W + 1, j0 + 256 + W - 1,
                 grad_keys=(j0, j0 + 256))
    sample_block(w, inp, gpu, 0, 0, 0, 300, 0, 300, grad_keys=None)
    sample_block(w, inp, gpu, 0, 3, w.Tq - 200, w.Tq, w.Tq - 200 - W + 1, w.Tq, grad_keys=(w.Tq - 200, w.Tq))


def test_encoder_mask_fwd_full():
    w = synth.WORKLOADS["encoder_mask"]
    inp = synth.make_inputs(w)
    gpu = run_gpu(w, inp)
    for b in (0, 5):
        for kvh in (0, 11):
            sample_block(w, inp, gpu, b, kvh, 0, w.Tq, 0, w.Tk)


@pytest.mark.parametrize("name", ["decode_lq1", "decode_lq4"])
def test_decode_full(name):
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    gpu = run_gpu(w, inp)
    for b, kvh in ((0, 0), (7, 3), (15, 7)):
        sample_block(w, inp, gpu, b, kvh, 0, w.Tq, 0, w.Tk)


def test_varlen_packed_fwd_bwd_full():
    """The bench's packed batch (8 causal sequences of U{256..2048} rows): whole
    shortest sequence and the tail of the longest, one KV group each."""
    w = synth.WORKLOADS["varlen_packed"]
    inp = synth.make_packed_inputs(w)
    dev = "cuda"
    cu = inp["cu"].to(device=dev, dtype=torch.int32)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    kw = dict(H=w.H, Hkv=w.Hkv, scale=w.scale, causal=True)
    o, lse = A.attn_varlen_fwd(q, k, v, cu, cu, w.Tq, w.Tk, **kw)
    dq, dk, dv = A.attn_varlen_bwd(q, k, v, o, do, lse, cu, cu, w.Tq, w.Tk, **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    G, hd = w.H // w.Hkv, w.hd
    lens = [int(x) for x in inp["lengths"]]
    cuh = [int(x) for x in inp["cu"]]
    for b, kvh, tail in ((int(np.argmin(lens)), 5, None), (int(np.argmax(lens)), 2, 128)):
        L, s0 = lens[b], cuh[b]
        r0 = 0 if tail is None else L - tail
        sl = lambda x, h0, h1: f64(x[s0:s0 + L, h0 * hd:h1 * hd])[None]
        qs = sl(inp["q"], kvh * G, (kvh + 1) * G)[:, r0:]
        ks, vs = sl(inp["k"], kvh, kvh + 1), sl(inp["v"], kvh, kvh + 1)
        okw = dict(H=G, Hkv=1, scale=w.scale, causal=True, q_offset=r0)
        o_ref, lse_ref = oracle.fwd(qs, ks, vs, **okw)
        og = o[s0 + r0:s0 + L, kvh * G * hd:(kvh + 1) * G * hd][None]
        lg = lse[b:b + 1, kvh * G:(kvh + 1) * G, r0:L]
        what = "varlen b%d kvh%d rows[%d,%d)" % (b, kvh, r0, L)
        compare_o_lse(og, lg, o_ref, lse_ref, w.dtype, what)
        dos = sl(inp["do"], kvh * G, (kvh + 1) * G)[:, r0:]
        gq, gk, gv = oracle.bwd(qs, ks, vs, dos, **okw)
        # dK/dV of the last `tail` keys are seen only by the sampled rows
        g0 = r0
        compare_grads((dq[s0 + r0:s0 + L, kvh * G * hd:(kvh + 1) * G * hd][None],
                       dk[s0 + g0:s0 + L, kvh * hd:(kvh + 1) * hd][None],
                       dv[s0 + g0:s0 + L, kvh * hd:(kvh + 1) * hd][None]),
                      (gq, gk[:, g0:], gv[:, g0:]), w.dtype, what)


@pytest.mark.parametrize("softcap", [0.0, 50.0], ids=["bias", "bias-softcap50"])
def test_bias_prefill_fwd_bwd_full(softcap):
    """The bench's biased GQA prefill: causal (window_right 0) with a [1, 1, T, T] fp32 bias,
    without and with a softcap (the cap applied to the score, then the bias)."""
    w = synth.WORKLOADS["gqa_prefill"]
    inp = synth.make_inputs(w)
    bias = synth.normal((1, 1, w.Tq, w.Tk), w.seed + 5, "f32")
    dev = "cuda"
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    kw = dict(H=w.H, Hkv=w.Hkv, scale=w.scale, window_left=-1, window_right=0, softcap=softcap)
    o, lse = A.attn_fwd_ex(q, k, v, bias=bias.to(dev), **kw)
    dq, dk, dv = A.attn_bwd_ex(q, k, v, o, do, lse, bias=bias.to(dev), **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    G, hd, T = w.H // w.Hkv, w.hd, w.Tq
    for b, kvh, r0 in ((1, 3, T - 128), (3, 6, 0)):
        r1 = r0 + 128
        qs = f64(inp["q"][b:b + 1, r0:r1, kvh * G * hd:(kvh + 1) * G * hd])
        ks = f64(inp["k"][b:b + 1, :r1, kvh * hd:(kvh + 1) * hd])
        vs = f64(inp["v"][b:b + 1, :r1, kvh * hd:(kvh + 1) * hd])
        bs = f64(bias[:, :, r0:r1, :r1])
        okw = dict(H=G, Hkv=1, scale=w.scale, window_left=-1, window_right=0, q_offset=r0, bias=bs,
                   softcap=softcap)
        o_ref, lse_ref = oracle.fwd_ex(qs, ks, vs, **okw)
        what = "bias b%d kvh%d rows[%d,%d)" % (b, kvh, r0, r1)
        compare_o_lse(o[b:b + 1, r0:r1, kvh * G * hd:(kvh + 1) * G * hd], lse[b:b + 1, kvh * G:(kvh + 1) * G, r0:r1],
                      o_ref, lse_ref, w.dtype, what)
        if r1 == T:  # keys [T-128, T) are seen only by the sampled rows
            dos = f64(inp["do"][b:b + 1, r0:r1, kvh * G * hd:(kvh + 1) * G * hd])
            gq, gk, gv = oracle.bwd_ex(qs, ks, vs, dos, **okw)
            compare_grads((dq[b:b + 1, r0:r1, kvh * G * hd:(kvh + 1) * G * hd], dk[b:b + 1, r0:r1, kvh * hd:(kvh + 1) * hd],
                           dv[b:b + 1, r0:r1, kvh * hd:(kvh + 1) * hd]),
                          (gq, gk[:, r0:r1], gv[:, r0:r1]), w.dtype, what)


def test_gqa_prefill_hd256_fwd_bwd_full():
    """hd 256 at its benchmark size: sampled blocks of two groups; the last 256 rows
    are every viewer of keys [T-256, T), so dK/dV there are exact."""
    w = synth.WORKLOADS["gqa_prefill_hd256"]
    inp = synth.make_inputs(w)
    gpu = run_gpu(w, inp)
    T = w.Tq
    sample_block(w, inp, gpu, 0, 0, 0, 200, 0, 200)
    sample_block(w, inp, gpu, 3, 3, T - 256, T, 0, T, grad_keys=(T - 256, T))
