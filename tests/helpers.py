"""Shared helpers for the GPU parity tests: build inputs, run the CUDA path
through the C ABI, run the fp64 oracle on the same rounded values, compare."""
import math

import numpy as np
import torch

import oracle
import attention_attn_fwd_08_gb300 as A
from attention_attn_fwd_08_gb300 import synth

# Tolerances: fp32 max-abs 1e-5 (rel 1e-4); 16-bit O max-abs 2e-2, LSE 1e-3,
# gradients 5e-2 relative Frobenius error against the oracle on the same
# rounded inputs.  fp32 gradients are held to 1e-4 relative Frobenius.
TOL = {
    "f32": dict(o=1e-5, lse=1e-5, grad=1e-4),
    "f16": dict(o=2e-2, lse=1e-3, grad=5e-2),
    "bf16": dict(o=2e-2, lse=1e-3, grad=5e-2),
}


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def make_mask(kind, B, Tk, seed):
    """None | 'shared' (one random 1/0 row) | 'batch' (prefix lengths) | 'holes' (random per batch,
    first keys masked so early causal rows see nothing) | 'band' (one unbroken run of kept keys
    per batch, starting past key 0 and ending before the last key)."""
    if kind is None:
        return None
    g = torch.Generator().manual_seed(seed)
    if kind == "shared":
        m = (torch.rand(Tk, generator=g) > 0.3).float()
        m[-1] = 1.0
        return m
    if kind == "batch":
        lens = synth.mask_lengths(B, max(1, Tk // 2), Tk, seed)
        return synth.prefix_mask(lens, Tk)
    if kind == "band":
        m = torch.zeros(B, Tk)
        for b in range(B):
            m[b, min(1 + 17 * b, Tk - 1):max(Tk - 3 - 5 * b, min(2 + 17 * b, Tk))] = 1.0
        return m
    if kind == "holes":
        m = (torch.rand(B, Tk, generator=g) > 0.4).float()
        m[:, : min(3, Tk)] = 0.0
        return m
    raise ValueError(kind)


def compare_o_lse(o_gpu, lse_gpu, o_ref, lse_ref, dt, what=""):
    tol = TOL[dt]
    og = f64(o_gpu)
    err = np.abs(og - o_ref).max() if og.size else 0.0
    assert np.isfinite(og).all(), what + ": non-finite O"
    assert err <= tol["o"], "%s: O max-abs %.3g > %.3g" % (what, err, tol["o"])
    if dt == "f32" and og.size:
        rel = np.linalg.norm(og - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
        assert rel <= 1e-4, "%s: O rel %.3g" % (what, rel)
    if lse_gpu is not None:
        lg = f64(lse_gpu)
        inf_g, inf_r = np.isneginf(lg), np.isneginf(lse_ref)
        assert (inf_g == inf_r).all(), what + ": -inf LSE rows differ"
        fin = ~inf_r
        if fin.any():
            e = np.abs(lg[fin] - lse_ref[fin]).max()
            assert e <= tol["lse"], "%s: LSE max-abs %.3g > %.3g" % (what, e, tol["lse"])


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    if nb == 0:
        return np.linalg.norm(a)
    return np.linalg.norm(a - b) / nb


def compare_grads(g_gpu, g_ref, dt, what=""):
    for name, g, r in zip(("dQ", "dK", "dV"), g_gpu, g_ref):
        gg = f64(g)
        assert np.isfinite(gg).all(), "%s: non-finite %s" % (what, name)
        e = rel_fro(gg, r)
        assert e <= TOL[dt]["grad"], "%s: %s rel-Frobenius %.3g > %.3g" % (what, name, e, TOL[dt]["grad"])


def inputs(dt, B, Tq, Tk, H, Hkv, hd, seed, backward=False):
    q = synth.normal((B, Tq, H * hd), seed, dt)
    k = synth.normal((B, Tk, Hkv * hd), seed + 1, dt)
    v = synth.normal((B, Tk, Hkv * hd), seed + 2, dt)
    do = synth.normal((B, Tq, H * hd), seed + 3, dt) if backward else None
    return q, k, v, do


def run_fwd_case(dt, B, Tq, Tk, H, Hkv, hd, causal=False, window=0, softcap=0.0, q_offset=0, mask=None,
                 backward=False, seed=1234, decode=False):
    q, k, v, do = inputs(dt, B, Tq, Tk, H, Hkv, hd, seed, backward)
    km = make_mask(mask, B, Tk, seed + 9)
    scale = 1.0 / math.sqrt(hd)
    kw = dict(H=H, Hkv=Hkv, scale=scale, causal=causal, window=window, softcap=softcap, q_offset=q_offset)
    dev = "cuda"
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    kmd = km.to(dev) if km is not None else None
    if decode:
        o, lse = A.attn_decode(qd, kd, vd, key_mask=kmd, **kw)
    else:
        o, lse = A.attn_fwd(qd, kd, vd, key_mask=kmd, **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    o_ref, lse_ref = oracle.fwd(f64(q), f64(k), f64(v), key_mask=None if km is None else f64(km), **kw)
    what = "%s B%d Tq%d Tk%d H%d/%d hd%d c%d w%d cap%g off%d mask=%s" % (dt, B, Tq, Tk, H, Hkv, hd, causal,
                                                                        window, softcap, q_offset, mask)
    compare_o_lse(o, lse, o_ref, lse_ref, dt, what)
    if backward:
        dod = do.to(dev)
        grads = A.attn_bwd(qd, kd, vd, o, dod, lse, key_mask=kmd, **kw)
        torch.cuda.synchronize()
        st, word = A.attn_get_device_status()
        assert st == A.OK, "device status word %#x" % word
        ref = oracle.bwd(f64(q), f64(k), f64(v), f64(do), key_mask=None if km is None else f64(km), **kw)
        compare_grads(grads, ref, dt, what)
