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
