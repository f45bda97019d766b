"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc and have no scratch buffer to hand over
(a plugin given only its inputs and outputs, a serving loop that forbids
allocation after start-up).  attn_decode_noalloc serves them from a fixed
32 MiB array inside the library.  These tests call it through the C ABI on
two calls in a row with different shapes (so a stale partial left by the first
call would show up in the second), for bf16 and fp16, and check each result
bit for bit against attn_decode (which takes a caller workspace but runs the
same kernels on the same split plan) and against the fp64 oracle within the
decode tolerances; and they check that a shape needing more scratch than the
array holds is refused before anything runs.

This file is collected last on purpose and passes both alone in a fresh
process and after the rest of the suite.
"""
import ctypes
import math

import pytest
import torch

import attention_attn_fwd_08_gb300 as A
from helpers import compare_o_lse, f64, inputs

pytestmark = pytest.mark.gpu


def noalloc_fn():
    L = A.lib()
    f = L.attn_decode_noalloc
    vp, i, fl, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
    f.argtypes = [i, vp, vp, vp, vp, vp, i, i, i, i, i, i, fl, i, i, fl, i, vp, ll, vp]
    f.restype = i
    return f


def run_noalloc(q, k, v, H, Hkv, q_offset, dt, softcap=0.0, window=0):
    B, Lq, hq = q.shape
    Tk = k.shape[1]
    hd = hq // H
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    code = {"bf16": 2, "f16": 1}[dt]
    st = noalloc_fn()(code, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Lq, Tk, H,
                      Hkv, hd, 1.0 / math.sqrt(hd), 1, window, softcap, q_offset, None, 0,
                      torch.cuda.current_stream().cuda_stream)
    assert st == A.OK, A.lib().attn_status_string(st)
    return o, lse


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_noalloc_decode_matches_workspace_decode_twice(dt, oracle):
    # two calls in a row with different shapes and flags: a partial left in the
    # shared array by the first call must not leak into the second
    calls = [(4, 4096, 16, 4, 3, dict(softcap=0.0, window=1000)), (1, 1500, 8, 2, 77, dict(softcap=30.0, window=0))]
    for Lq, Tk, H, Hkv, seed, kw in calls:
        B, hd = 3, 128
        q, k, v, _ = inputs(dt, B, Lq, Tk, H, Hkv, hd, seed)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o_ws, lse_ws = A.attn_decode(qd, kd, vd, H=H, Hkv=Hkv, causal=True, q_offset=Tk - Lq, **kw)
        o, lse = run_noalloc(qd, kd, vd, H, Hkv, Tk - Lq, dt, **kw)
        torch.cuda.synchronize()
        st, word = A.attn_get_device_status()
        assert st == A.OK, "device status word %#x" % word
        # same kernels on the same split plan: the results agree bit for bit
        assert torch.equal(o, o_ws) and torch.equal(lse, lse_ws)
        # and both match the fp64 oracle within the decode tolerances
        o_ref, lse_ref = oracle.fwd(f64(q), f64(k), f64(v), H=H, Hkv=Hkv, scale=1.0 / math.sqrt(hd), causal=True,
                                    q_offset=Tk - Lq, **kw)
        compare_o_lse(o, lse, o_ref, lse_ref, dt, "noalloc %s Lq%d Tk%d" % (dt, Lq, Tk))


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # B=64, Lq=16, H=64, Hkv=16, hd=128 needs about 34 MB of partials (> 32 MiB)
    assert A.attn_decode_workspace_size(64, 16, 32768, 64, 16, 128) > 32 << 20
    bad = 0x1000  # never dereferenced: the size check refuses the call first
    st = noalloc_fn()(2, bad, bad, bad, bad, None, 64, 16, 32768, 64, 16, 128, 0.088, 1, 0, 0.0, 32752, None, 0,
                      None)
    assert st == A.ERR_UNSUPPORTED
