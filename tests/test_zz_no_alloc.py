"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc and have no scratch buffer to hand over
(a plugin given only its inputs and outputs, a serving loop that forbids
allocation after start-up).  attn_decode_noalloc serves them from a fixed
32 MiB array inside the library.  These tests call it through the C ABI and
check it against attn_decode, which takes a caller workspace, on two calls in
a row with different shapes (so a stale partial left by the first call would
show up in the second), and check that a shape needing more scratch than the
array holds is refused before anything runs.

This file is collected last on purpose and passes both alone in a fresh
process and after the rest of the suite.
"""
import ctypes
import math

import pytest
import torch

import attention_attn_fwd_08_gb300 as A
from helpers import TOL, inputs

pytestmark = pytest.mark.gpu


def noalloc_fn():
    L = A.lib()
    f = L.attn_decode_noalloc
    vp, i, fl, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
    f.argtypes = [i, vp, vp, vp, vp, vp, i, i, i, i, i, i, fl, i, i, fl, i, vp, ll, vp]
    f.restype = i
    return f


def run_noalloc(q, k, v, H, Hkv, q_offset, softcap=0.0, window=0):
    B, Lq, hq = q.shape
    Tk = k.shape[1]
    hd = hq // H
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    st = noalloc_fn()(2, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Lq, Tk, H, Hkv,
                      hd, 1.0 / math.sqrt(hd), 1, window, softcap, q_offset, None, 0,
                      torch.cuda.current_stream().cuda_stream)
    assert st == A.OK, A.lib().attn_status_string(st)
    return o, lse


@pytest.mark.parametrize("first,second", [((4, 4096, 16, 4, 3), (1, 1500, 8, 2, 77))])
def test_noalloc_decode_matches_workspace_decode_twice(first, second):
    for call, (Lq, Tk, H, Hkv, seed) in enumerate((first, second)):
        B, hd = 3, 128
        q, k, v, _ = inputs("bf16", B, Lq, Tk, H, Hkv, hd, seed)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        kw = dict(softcap=30.0 if call else 0.0, window=0 if call else 1000)
        o_ref, lse_ref = A.attn_decode(qd, kd, vd, H=H, Hkv=Hkv, causal=True, q_offset=Tk - Lq, **kw)
        o, lse = run_noalloc(qd, kd, vd, H, Hkv, Tk - Lq, **kw)
        torch.cuda.synchronize()
        st, word = A.attn_get_device_status()
        assert st == A.OK, "device status word %#x" % word
        tol = TOL["bf16"]
        assert (o.float() - o_ref.float()).abs().max().item() <= tol["o"]
        assert (lse - lse_ref).abs().max().item() <= tol["lse"]


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # B=64, Lq=16, H=64, Hkv=16, hd=128 needs about 34 MB of partials (> 32 MiB)
    assert A.attn_decode_workspace_size(64, 16, 32768, 64, 16, 128) > 32 << 20
    bad = 0x1000  # never dereferenced: the size check refuses the call first
    st = noalloc_fn()(2, bad, bad, bad, bad, None, 64, 16, 32768, 64, 16, 128, 0.088, 1, 0, 0.0, 32752, None, 0,
                      None)
    assert st == A.ERR_UNSUPPORTED
