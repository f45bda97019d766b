"""Rotary embedding on the GPU against the fp64 oracle (ferrotensor
engine/attention.rs, rope / rope_theta), every dtype, several head sizes,
positions far from 0; and its composition with attention (the scores of
rotated q and k depend on relative positions only)."""
import numpy as np
import pytest
import torch

import oracle
import attention_attn_fwd_08_gb300 as A
from attention_attn_fwd_08_gb300 import synth
from helpers import f64

pytestmark = pytest.mark.gpu

# max-abs error allowed on N(0,1) inputs: rounding of the output dtype (16-bit also the fp32 angle)
TOL = {"f32": 2e-5, "f16": 4e-3, "bf16": 2.5e-2}


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("hd,H,pos,theta", [(128, 8, 0, 10000.0), (64, 4, 5000, 10000.0), (256, 2, 31, 500000.0),
                                            (32, 3, 7, 10000.0)])
def test_rope_matches_oracle(dt, hd, H, pos, theta):
    x = synth.normal((2, 300, H * hd), 900 + hd, dt)
    y = A.attn_rope(x.cuda(), H=H, pos=pos, theta=theta)
    torch.cuda.synchronize()
    ref = oracle.rope(f64(x), head_dim=hd, pos=pos, theta=theta)
    err = np.abs(f64(y) - ref).max()
    assert err <= TOL[dt], (dt, hd, err)


def test_rope_then_attention_depends_on_relative_position():
    """Attention over RoPE'd q and k is the same whatever the common offset."""
    H, Hkv, hd, T = 4, 2, 64, 200
    q = synth.normal((1, T, H * hd), 910, "f32").cuda()
    k = synth.normal((1, T, Hkv * hd), 911, "f32").cuda()
    v = synth.normal((1, T, Hkv * hd), 912, "f32").cuda()
    outs = []
    for pos in (0, 1000):
        qr = A.attn_rope(q.clone(), H=H, pos=pos)
        kr = A.attn_rope(k.clone(), H=Hkv, pos=pos)
        outs.append(A.attn_fwd(qr, kr, v, H=H, Hkv=Hkv, causal=True)[0])
    torch.cuda.synchronize()
    assert torch.allclose(outs[0], outs[1], atol=2e-4)


# ------------------------------------------------------------ fused rotation
def _turned(x, H, hd, pos, theta, dt):
    """The oracle's rotary turn of x at positions pos + s, rounded to dt like the
    16-bit operands the kernels read (fp64 otherwise)."""
    r = oracle.rope(f64(x), head_dim=hd, pos=pos, theta=theta)
    return r if dt == "f32" else f64(torch.from_numpy(r).to(synth.DTYPES[dt]))


def _turn_back(g, H, hd, pos, theta):
    """R^T g, the inverse turn, through the oracle's turn: R(-t) = S R(t) S with S
    negating the second half of every head vector."""
    B, T, C = g.shape
    s = np.ones(hd)
    s[hd // 2:] = -1.0
    S = np.tile(s, C // hd)
    return oracle.rope(g * S, head_dim=hd, pos=pos, theta=theta) * S


ROPE_CASES = [
    dict(dt="bf16", hd=128, causal=True, q_offset=0, rope_pos=0),
    dict(dt="bf16", hd=128, causal=True, window=150, softcap=30.0, q_offset=64, rope_pos=1000),
    dict(dt="f16", hd=64, causal=False, mask="batch", q_offset=0, rope_pos=7),
    dict(dt="bf16", hd=96, causal=True, q_offset=20, rope_pos=3),   # q turned into the workspace
    dict(dt="f32", hd=64, causal=True, q_offset=0, rope_pos=0),
]


@pytest.mark.parametrize("case", ROPE_CASES, ids=lambda c: "-".join("%s%s" % kv for kv in c.items()))
def test_fwd_rope_equals_rope_then_fwd_and_oracle(case):
    from helpers import compare_o_lse, make_mask
    case = dict(case)
    dt, hd, rope_pos, q_offset = case.pop("dt"), case.pop("hd"), case.pop("rope_pos"), case.pop("q_offset")
    mask = case.pop("mask", None)
    B, Tq, H, Hkv, theta = 2, 300, 4, 2, 10000.0
    Tk = Tq + q_offset
    q = synth.normal((B, Tq, H * hd), 930 + hd, dt)
    k = synth.normal((B, Tk, Hkv * hd), 931 + hd, dt)
    v = synth.normal((B, Tk, Hkv * hd), 932 + hd, dt)
    km = make_mask(mask, B, Tk, 933)
    kw = dict(H=H, Hkv=Hkv, q_offset=q_offset, key_mask=None if km is None else km.cuda(), **case)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = A.attn_fwd_rope(qd, kd, vd, rope_pos=rope_pos, rope_theta=theta, **kw)
    # the same through the standalone turn
    qr = A.attn_rope(qd.clone(), H=H, pos=rope_pos + q_offset, theta=theta)
    kr = A.attn_rope(kd.clone(), H=Hkv, pos=rope_pos, theta=theta)
    o2, lse2 = A.attn_fwd(qr, kr, vd, **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    assert torch.equal(qd, q.cuda()) and torch.equal(kd, k.cuda()), "q and k must be left unrotated"
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    # and against the oracle on the turned operands
    qt = _turned(q, H, hd, rope_pos + q_offset, theta, dt)
    kt = _turned(k, Hkv, hd, rope_pos, theta, dt)
    o_ref, lse_ref = oracle.fwd(qt, kt, f64(v), H=H, Hkv=Hkv, scale=1.0 / np.sqrt(hd), q_offset=q_offset,
                                key_mask=None if km is None else f64(km), **case)
    compare_o_lse(o, lse, o_ref, lse_ref, dt, "fwd_rope %s hd%d" % (dt, hd))


@pytest.mark.parametrize("case", ROPE_CASES, ids=lambda c: "-".join("%s%s" % kv for kv in c.items()))
def test_bwd_rope_gradients_of_unrotated_inputs(case):
    from helpers import compare_grads, make_mask
    case = dict(case)
    dt, hd, rope_pos, q_offset = case.pop("dt"), case.pop("hd"), case.pop("rope_pos"), case.pop("q_offset")
    mask = case.pop("mask", None)
    B, Tq, H, Hkv, theta = 2, 260, 4, 2, 10000.0
    Tk = Tq + q_offset
    q = synth.normal((B, Tq, H * hd), 940 + hd, dt)
    k = synth.normal((B, Tk, Hkv * hd), 941 + hd, dt)
    v = synth.normal((B, Tk, Hkv * hd), 942 + hd, dt)
    do = synth.normal((B, Tq, H * hd), 943 + hd, dt)
    km = make_mask(mask, B, Tk, 944)
    kw = dict(H=H, Hkv=Hkv, q_offset=q_offset, key_mask=None if km is None else km.cuda(), rope_pos=rope_pos,
              rope_theta=theta, **case)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = A.attn_fwd_rope(qd, kd, vd, **kw)
    dq, dk, dv = A.attn_bwd_rope(qd, kd, vd, o, dod, lse, **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    qt = _turned(q, H, hd, rope_pos + q_offset, theta, dt)
    kt = _turned(k, Hkv, hd, rope_pos, theta, dt)
    ok = dict(H=H, Hkv=Hkv, scale=1.0 / np.sqrt(hd), q_offset=q_offset, key_mask=None if km is None else f64(km),
              **case)
    gq, gk, gv = oracle.bwd(qt, kt, f64(v), f64(do), **ok)
    ref = (_turn_back(gq, H, hd, rope_pos + q_offset, theta), _turn_back(gk, Hkv, hd, rope_pos, theta), gv)
    compare_grads((dq, dk, dv), ref, dt, "bwd_rope %s hd%d" % (dt, hd))
