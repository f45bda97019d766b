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
