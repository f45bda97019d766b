"""Packed variable-length attention on the GPU against the fp64 oracle
(brotensor ops/flash_attention.h, flash_attention_varlen_forward / _backward):
ragged and empty sequences, lengths off every tile boundary, sequences longer
than a 256-row work item, query and key lengths that differ, GQA, window and
softcap, both kernel families.  Rows outside every sequence must keep what the
caller left there.  Every call goes through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_attn_fwd_08_gb300 as A
from attention_attn_fwd_08_gb300 import synth
from helpers import TOL, compare_grads, f64

pytestmark = pytest.mark.gpu

SENTINEL = 3.0


def cu_of(lengths):
    return [0] + list(np.cumsum(lengths))


def packed_inputs(dt, cu_q, cu_k, H, Hkv, hd, seed, pad_q=5, pad_k=3):
    tq, tk = cu_q[-1] + pad_q, cu_k[-1] + pad_k  # rows past the last sequence belong to none
    q = synth.normal((tq, H * hd), seed, dt)
    k = synth.normal((tk, Hkv * hd), seed + 1, dt)
    v = synth.normal((tk, Hkv * hd), seed + 2, dt)
    do = synth.normal((tq, H * hd), seed + 3, dt)
    return q, k, v, do


def run_varlen(dt, lens_q, lens_k, H, Hkv, hd, seed, backward=True, **flags):
    cu_q, cu_k = cu_of(lens_q), cu_of(lens_k)
    q, k, v, do = packed_inputs(dt, cu_q, cu_k, H, Hkv, hd, seed)
    kw = dict(H=H, Hkv=Hkv, scale=1.0 / math.sqrt(hd), **flags)
    mq, mk = max(lens_q), max(lens_k)
    dev = "cuda"
    cq = torch.tensor(cu_q, dtype=torch.int32, device=dev)
    ck = torch.tensor(cu_k, dtype=torch.int32, device=dev)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o = torch.full_like(qd, SENTINEL)
    lse = torch.full((len(lens_q), H, mq), 5.0, dtype=torch.float32, device=dev)
    A.attn_varlen_fwd(qd, kd, vd, cq, ck, mq, mk, o=o, lse=lse, **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    o_ref, lse_ref = oracle.varlen_fwd(f64(q), f64(k), f64(v), cu_q, cu_k, **kw)
    what = "%s lens_q=%s lens_k=%s H%d/%d hd%d %s" % (dt, lens_q, lens_k, H, Hkv, hd, flags)
    og = f64(o)
    inside = np.zeros(og.shape[0], bool)
    inside[: cu_q[-1]] = True
    assert (og[~inside] == SENTINEL).all(), what + ": rows outside every sequence were written"
    assert np.isfinite(og).all()
    err = np.abs(og[inside] - o_ref[inside]).max()
    assert err <= TOL[dt]["o"], "%s: O max-abs %.3g" % (what, err)
    lg = f64(lse)
    for b, lr in enumerate(lse_ref):
        n = lr.shape[1]
        got = lg[b, :, :n]
        assert (np.isneginf(got) == np.isneginf(lr)).all(), what + ": -inf LSE rows differ"
        fin = ~np.isneginf(lr)
        if fin.any():
            assert np.abs(got[fin] - lr[fin]).max() <= TOL[dt]["lse"], what + ": LSE"
    if not backward:
        return
    dq = torch.full_like(qd, SENTINEL)
    dk = torch.full_like(kd, SENTINEL)
    dv = torch.full_like(vd, SENTINEL)
    A.attn_varlen_bwd(qd, kd, vd, o, dod, lse, cq, ck, mq, mk, dq=dq, dk=dk, dv=dv, **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    ref = oracle.varlen_bwd(f64(q), f64(k), f64(v), f64(do), cu_q, cu_k, **kw)
    kin = np.zeros(dk.shape[0], bool)
    kin[: cu_k[-1]] = True
    assert (f64(dq)[~inside] == SENTINEL).all() and (f64(dk)[~kin] == SENTINEL).all() \
        and (f64(dv)[~kin] == SENTINEL).all(), what + ": gradient rows outside every sequence were written"
    compare_grads((dq[: cu_q[-1]], dk[: cu_k[-1]], dv[: cu_k[-1]]),
                  (ref[0][: cu_q[-1]], ref[1][: cu_k[-1]], ref[2][: cu_k[-1]]), dt, what)


# ragged, an empty sequence, one row, a 256-row item boundary, several items
LENS = [300, 0, 129, 1, 520, 64, 257]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("flags", [dict(causal=True), dict(causal=False), dict(causal=True, window=100, softcap=30.0)],
                         ids=["causal", "full", "window-softcap"])
def test_varlen_16bit(dt, hd, flags):
    run_varlen(dt, LENS, LENS, 4, 2, hd, seed=700 + hd, **flags)


def test_varlen_query_and_key_lengths_differ():
    """Non-causal cross attention: every sequence has its own query and key counts."""
    run_varlen("bf16", [70, 0, 200, 33], [150, 40, 0, 333], 8, 2, 128, seed=720, causal=False)


def test_varlen_many_items_per_cta():
    """More (sequence, head, 256-row block) items than SMs: every persistent CTA runs
    several sequences back to back."""
    lens = [int(x) for x in np.random.default_rng(5).integers(1, 700, size=24)]
    run_varlen("bf16", lens, lens, 16, 4, 128, seed=730, causal=True)


def test_varlen_more_sequences_than_a_warp():
    """Up to 32 sequences, the forward deals out only the query blocks that hold rows;
    with more it numbers every sequence's blocks up to the longest (the surplus ones
    empty).  Both numberings must cover every row exactly once."""
    lens = [int(x) for x in np.random.default_rng(6).integers(0, 400, size=40)]
    lens[7] = 600
    run_varlen("bf16", lens, lens, 4, 2, 128, seed=735, backward=False, causal=True)
    run_varlen("bf16", lens[:32], lens[:32], 4, 2, 128, seed=736, backward=False, causal=True)


@pytest.mark.parametrize("hd", [64, 128])
def test_varlen_fp32(hd):
    run_varlen("f32", [40, 0, 97, 1, 130], [40, 0, 97, 1, 130], 2, 1, hd, seed=740, causal=True, window=50)


def test_varlen_one_sequence_equals_dense():
    """A single packed sequence is the dense call with B = 1."""
    H, Hkv, hd, T = 8, 2, 128, 333
    q, k, v, do = packed_inputs("bf16", [0, T], [0, T], H, Hkv, hd, seed=750, pad_q=0, pad_k=0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    o1, l1 = A.attn_varlen_fwd(qd, kd, vd, cu, cu, T, T, H=H, Hkv=Hkv, causal=True)
    o2, l2 = A.attn_fwd(qd[None], kd[None], vd[None], H=H, Hkv=Hkv, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[0]) and torch.equal(l1, l2)


def test_varlen_bounds_violation_is_reported_and_clipped():
    """A sequence longer than max_seqlen_q is cut to the bound; no row past the bound
    or past the tensor is written, and the status call reports invalid input."""
    H, Hkv, hd = 2, 1, 64
    q, k, v, _ = packed_inputs("bf16", [0, 100], [0, 100], H, Hkv, hd, seed=760, pad_q=0, pad_k=0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    cu = torch.tensor([0, 100], dtype=torch.int32, device="cuda")
    o = torch.full_like(qd, SENTINEL)
    A.attn_varlen_fwd(qd, kd, vd, cu, cu, 64, 100, H=H, Hkv=Hkv, causal=True, o=o)
    st, word = A.attn_get_device_status()
    assert st == A.ERR_INVALID_ARG and word == (1 << 9), (st, hex(word))
    assert (f64(o)[64:] == SENTINEL).all()
    o_ref, _ = oracle.varlen_fwd(f64(q), f64(k), f64(v), [0, 64], [0, 100], H=H, Hkv=Hkv, scale=1 / 8.0, causal=True)
    assert np.abs(f64(o)[:64] - o_ref[:64]).max() <= 2e-2
    # cu_seqlens past the tensor's rows: cut at the tensor's end
    cu2 = torch.tensor([0, 150], dtype=torch.int32, device="cuda")
    A.attn_varlen_fwd(qd, kd, vd, cu2, cu2, 100, 100, H=H, Hkv=Hkv, causal=True, o=o)
    st, word = A.attn_get_device_status()
    assert st == A.ERR_INVALID_ARG
    st, word = A.attn_get_device_status()
    assert st == A.OK
