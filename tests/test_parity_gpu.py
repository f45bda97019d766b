"""GPU parity against the fp64 oracle at sizes the oracle finishes in seconds,
spanning several 128-row tiles with ragged tails, every masking feature and
the degenerate cases.  Every call goes through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_attn_fwd_08_gb300 as A
from helpers import compare_o_lse, f64, inputs, run_fwd_case

pytestmark = pytest.mark.gpu

FWD_FLAGS = [
    dict(causal=False),
    dict(causal=True),
    dict(causal=True, window=100),
    dict(causal=True, window=37, softcap=50.0),
    dict(causal=False, softcap=5.0, mask="batch"),
    dict(causal=False, window=64, mask="shared"),
    dict(causal=True, mask="holes"),          # early rows fully masked
    dict(causal=False, mask="band"),          # key tiles inside an unbroken kept run read no mask
    dict(causal=True, q_offset=77, window=150),
]


# hd 32 and 96 run the 64 / 128 tensor-core kernels with the columns past the head
# read as zeros (4-D maps) and never written
@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("hd", [32, 64, 96, 128])
@pytest.mark.parametrize("flags", FWD_FLAGS, ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_fwd_16bit(dt, hd, flags):
    Tq = 300
    Tk = Tq + flags.get("q_offset", 0)
    run_fwd_case(dt, 2, Tq, Tk, 4, 2, hd, seed=100 + hd, **flags)


@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("flags", FWD_FLAGS[:4] + FWD_FLAGS[6:], ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_fwd_fp32(hd, flags):
    Tq = 200
    Tk = Tq + flags.get("q_offset", 0)
    run_fwd_case("f32", 1, Tq, Tk, 2, 1, hd, seed=200 + hd, **flags)


# More work items (256-row query blocks x heads x batch) than the GPU has SMs, so
# every CTA of the persistent forward runs several items back to back with
# different key ranges, masks and tile activity.
MULTI_ITEM_FLAGS = [
    dict(causal=True),
    dict(causal=True, window=200, softcap=30.0),
    dict(causal=False, mask="holes"),
    dict(causal=False, mask="band"),
    dict(causal=True, q_offset=100, window=300),
]


@pytest.mark.parametrize("flags", MULTI_ITEM_FLAGS, ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_fwd_many_items_per_cta(flags):
    Tq = 520  # 3 query blocks, the last one ragged (8 rows, tile B empty)
    Tk = Tq + flags.get("q_offset", 0)
    run_fwd_case("bf16", 4, Tq, Tk, 32, 8, 128, seed=150, **flags)


def test_fwd_many_items_hd64_f16():
    run_fwd_case("f16", 3, 700, 700, 24, 4, 64, causal=True, window=333, seed=151)


def test_fp32_causal_workload_full():
    """B=1, H=Hkv=1, T=128, hd=64, scale=1/8, causal, fp32."""
    run_fwd_case("f32", 1, 128, 128, 1, 1, 64, causal=True, seed=0x5EED0001)


BWD_FLAGS = [
    dict(causal=True),
    dict(causal=False, mask="batch"),
    dict(causal=True, window=90, softcap=50.0),
    dict(causal=True, mask="holes", softcap=3.0),
    dict(causal=True, q_offset=40, window=130),
]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("hd", [32, 64, 96, 128])
@pytest.mark.parametrize("flags", BWD_FLAGS, ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_bwd_16bit(dt, hd, flags):
    Tq = 260
    Tk = Tq + flags.get("q_offset", 0)
    run_fwd_case(dt, 2, Tq, Tk, 4, 2, hd, backward=True, seed=300 + hd, **flags)


# More dQ work items (128-row query blocks x heads x batch) than SMs: every CTA of
# the persistent dQ kernel runs several items with different key ranges.
@pytest.mark.parametrize("flags", [dict(causal=True), dict(causal=True, window=150, softcap=20.0),
                                   dict(causal=False, mask="holes")],
                         ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_bwd_many_items_per_cta(flags):
    run_fwd_case("bf16", 4, 300, 300, 32, 8, 128, backward=True, seed=310, **flags)


@pytest.mark.parametrize("dt,hd", [("bf16", 128), ("f16", 64)])
def test_softcap_polynomial_and_fallback_mix(dt, hd):
    """A softcap of 8 puts about one raw score q.k in 10^4 outside the range of the
    kernels' tanh polynomial (|q.k| * scale / softcap > 1/2), so within one call
    some warps' tiles take the exp-based tanh and the rest the polynomial."""
    run_fwd_case(dt, 2, 390, 390, 4, 2, hd, backward=True, causal=True, window=300, softcap=8.0, seed=320)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("hd", [64, 128])
def test_softcap_three_tiers(dt, hd):
    """The forward picks, per warp and key tile, the short tanh polynomial (every
    |scale*q.k/softcap| <= 1/8), the cubic one (<= 1/2) or the exp-based tanh.
    With softcap 30 about half the warps' tiles of N(0,1) data fit the short one,
    and a few query rows scaled by 8 push their warps past the cubic's range: the
    input check below confirms that one call meets all three."""
    B, T, H, Hkv, cap = 1, 384, 2, 1, 30.0
    q, k, v, _ = inputs(dt, B, T, T, H, Hkv, hd, seed=330)
    q[:, 300:304] = (q[:, 300:304].float() * 8).to(q.dtype)
    scale = 1.0 / math.sqrt(hd)
    y = np.einsum("bihd,bjhd->bhij", f64(q).reshape(B, T, H, hd),
                  np.repeat(f64(k).reshape(B, T, Hkv, hd), H // Hkv, axis=2)) * scale / cap
    tiers = set()
    for h in range(H):
        for i0 in range(0, T, 32):             # one warp's 32 rows
            for j0 in range(0, i0 + 32, 128):  # the key tiles of its 128-row query tile
                a = np.abs(y[:, h, i0:i0 + 32, j0:j0 + 128]).max()
                tiers.add(0 if a <= 0.125 else 1 if a <= 0.5 else 2)
    assert tiers == {0, 1, 2}, tiers
    kw = dict(H=H, Hkv=Hkv, scale=scale, causal=True, softcap=cap)
    o, lse = A.attn_fwd(q.cuda(), k.cuda(), v.cuda(), **kw)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    o_ref, lse_ref = oracle.fwd(f64(q), f64(k), f64(v), **kw)
    compare_o_lse(o, lse, o_ref, lse_ref, dt, "softcap tiers %s hd%d" % (dt, hd))


@pytest.mark.parametrize("flags", BWD_FLAGS[:3], ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_bwd_fp32(flags):
    Tq = 150
    Tk = Tq + flags.get("q_offset", 0)
    run_fwd_case("f32", 1, Tq, Tk, 2, 1, 64, backward=True, seed=400, **flags)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("Lq,H,Hkv", [(1, 8, 2), (4, 8, 2), (16, 4, 4), (4, 32, 8), (3, 12, 1)])
@pytest.mark.parametrize("hd", [64, 128, 256])
def test_decode(dt, Lq, H, Hkv, hd):
    Tk = 1000
    run_fwd_case(dt, 3, Lq, Tk, H, Hkv, hd, causal=True, q_offset=Tk - Lq, decode=True, seed=500 + Lq)


@pytest.mark.parametrize("flags", [dict(window=200), dict(softcap=30.0, mask="holes"), dict(mask="shared"),
                                   dict(window=5000, softcap=1.0)],
                         ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_decode_features(flags):
    Tk, Lq = 3333, 4
    run_fwd_case("bf16", 2, Lq, Tk, 8, 2, 128, causal=True, q_offset=Tk - Lq, decode=True, seed=600, **flags)


def _decode_len_reference(q, k, v, lengths, H, Hkv, hd, km=None, **flags):
    """Per sequence b: the oracle on its first L_b keys, query rows at positions
    L_b - Lq .. L_b - 1 (rows at negative positions see nothing: O = 0, LSE = -inf)."""
    B, Lq = q.shape[0], q.shape[1]
    o_ref = np.zeros((B, Lq, H * hd))
    lse_ref = np.full((B, H, Lq), -np.inf)
    for b in range(B):
        L = int(lengths[b])
        first = max(Lq - L, 0)  # first query row at a position >= 0
        if L == 0 or first >= Lq:
            continue
        kb = f64(k[b:b + 1, :L])
        vb = f64(v[b:b + 1, :L])
        mb = None if km is None else f64(km[b:b + 1, :L])
        o_b, l_b = oracle.fwd(f64(q[b:b + 1, first:]), kb, vb, H=H, Hkv=Hkv, scale=1.0 / math.sqrt(hd), causal=True,
                              q_offset=L - Lq + first, key_mask=mb, **flags)
        o_ref[b, first:] = o_b[0]
        lse_ref[b, :, first:] = l_b[0]
    return o_ref, lse_ref


@pytest.mark.parametrize("flags", [dict(), dict(window=300, softcap=25.0), dict(mask=True)],
                         ids=["plain", "window-softcap", "keymask"])
def test_decode_len_matches_oracle(flags):
    """Device-resident lengths, including L < Lq and L = 0, against the oracle."""
    from helpers import compare_o_lse, make_mask
    B, Lq, Tk, H, Hkv, hd = 6, 4, 700, 8, 2, 128
    q, k, v, _ = inputs("bf16", B, Lq, Tk, H, Hkv, hd, 905)
    lengths = torch.tensor([700, 333, 4, 2, 0, 65], dtype=torch.int32)
    flags = dict(flags)
    km = make_mask("batch", B, Tk, 906) if flags.pop("mask", False) else None
    o, lse = A.attn_decode_len(q.cuda(), k.cuda(), v.cuda(), lengths.cuda(), H=H, Hkv=Hkv,
                               key_mask=None if km is None else km.cuda(), **flags)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    o_ref, lse_ref = _decode_len_reference(q, k, v, lengths, H, Hkv, hd, km=km, **flags)
    compare_o_lse(o, lse, o_ref, lse_ref, "bf16", "decode_len %s" % flags)


def test_decode_len_hd256_window_softcap():
    from helpers import compare_o_lse
    B, Lq, Tk, H, Hkv, hd = 3, 2, 900, 4, 2, 256
    q, k, v, _ = inputs("f16", B, Lq, Tk, H, Hkv, hd, 908)
    lengths = torch.tensor([900, 411, 1], dtype=torch.int32)
    o, lse = A.attn_decode_len(q.cuda(), k.cuda(), v.cuda(), lengths.cuda(), H=H, Hkv=Hkv, window=200, softcap=30.0)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    o_ref, lse_ref = _decode_len_reference(q, k, v, lengths, H, Hkv, hd, window=200, softcap=30.0)
    compare_o_lse(o, lse, o_ref, lse_ref, "f16", "decode_len hd256")


def test_decode_len_graph_replay_follows_lengths():
    """One captured launch, replayed after the device lengths change, matches the
    oracle for each set of lengths."""
    from helpers import compare_o_lse
    B, Lq, Tk, H, Hkv, hd = 3, 2, 1500, 8, 2, 128
    q, k, v, _ = inputs("bf16", B, Lq, Tk, H, Hkv, hd, 907)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    lengths = torch.tensor([100, 100, 100], dtype=torch.int32, device="cuda")
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, Lq), dtype=torch.float32, device="cuda")
    ws = torch.empty(A.attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first call outside the capture (one-time set-up)
        A.attn_decode_len(qd, kd, vd, lengths, H=H, Hkv=Hkv, o=o, lse=lse, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        A.attn_decode_len(qd, kd, vd, lengths, H=H, Hkv=Hkv, o=o, lse=lse, workspace=ws)
    for lens in ([1500, 777, 1], [64, 1499, 300]):
        lengths.copy_(torch.tensor(lens, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        st, word = A.attn_get_device_status()
        assert st == A.OK, "device status word %#x" % word
        o_ref, lse_ref = _decode_len_reference(q, k, v, lens, H, Hkv, hd)
        compare_o_lse(o, lse, o_ref, lse_ref, "bf16", "graph replay lengths %s" % lens)


def test_decode_short_cache_and_noncausal():
    run_fwd_case("bf16", 2, 2, 7, 4, 2, 64, causal=True, q_offset=5, decode=True, seed=700)
    run_fwd_case("f16", 2, 2, 130, 4, 2, 64, causal=False, q_offset=0, decode=True, seed=701)


def test_decode_fp32_routes_to_fp32_kernel():
    run_fwd_case("f32", 1, 4, 300, 4, 2, 64, causal=True, q_offset=296, decode=True, seed=702)


# ------------------------------------------------------------ edge cases
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_single_query_single_key(dt):
    run_fwd_case(dt, 1, 1, 1, 2, 1, 64, causal=True, backward=True, seed=800)


def test_ragged_small_and_tq_ne_tk():
    run_fwd_case("bf16", 3, 7, 5, 2, 2, 128, causal=False, seed=801)
    run_fwd_case("bf16", 1, 129, 257, 2, 1, 64, causal=True, q_offset=128, backward=True, seed=802)
    run_fwd_case("f16", 1, 5, 300, 2, 1, 64, causal=False, backward=True, seed=803)


def test_window_larger_than_sequence_equals_unbounded():
    q, k, v, _ = inputs("bf16", 1, 200, 200, 2, 1, 128, 900)
    a, la = A.attn_fwd(q.cuda(), k.cuda(), v.cuda(), H=2, Hkv=1, causal=True, window=0)
    b, lb = A.attn_fwd(q.cuda(), k.cuda(), v.cuda(), H=2, Hkv=1, causal=True, window=500)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_softcap_zero_is_off_on_gpu():
    q, k, v, _ = inputs("bf16", 1, 150, 150, 2, 1, 64, 901)
    a, la = A.attn_fwd(q.cuda(), k.cuda(), v.cuda(), H=2, Hkv=1, causal=True)
    b, lb = A.attn_fwd(q.cuda(), k.cuda(), v.cuda(), H=2, Hkv=1, causal=True, softcap=0.0)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_no_keys_gives_zero_output_and_neg_inf_lse():
    q = torch.randn(2, 5, 2 * 64, device="cuda").bfloat16()
    k = torch.empty(2, 0, 64, device="cuda", dtype=torch.bfloat16)
    o, lse = A.attn_fwd(q, k, k, H=2, Hkv=1)
    torch.cuda.synchronize()
    assert (o == 0).all() and torch.isneginf(lse).all()
    o, lse = A.attn_decode(q[:, :1].contiguous(), k, k, H=2, Hkv=1, q_offset=0)
    torch.cuda.synchronize()
    assert (o == 0).all() and torch.isneginf(lse).all()


def test_empty_batch_is_noop():
    q = torch.empty(0, 4, 128, device="cuda", dtype=torch.bfloat16)
    o = torch.full_like(q, 3.0)
    A.attn_fwd(q, q, q, H=1, Hkv=1, o=o)
    torch.cuda.synchronize()


def test_outputs_are_overwritten_not_accumulated():
    q, k, v, do = inputs("bf16", 1, 140, 140, 2, 1, 64, 902, backward=True)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = A.attn_fwd(qd, kd, vd, H=2, Hkv=1, causal=True)
    g1 = A.attn_bwd(qd, kd, vd, o, dod, lse, H=2, Hkv=1, causal=True)
    g1 = [t.clone() for t in g1]
    dq, dk, dv = (torch.full_like(t, 7.0) for t in g1)
    g2 = A.attn_bwd(qd, kd, vd, o, dod, lse, H=2, Hkv=1, causal=True, dq=dq, dk=dk, dv=dv)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_bwd_passes_run_separately():
    """dQ (pass 4) then dK/dV (pass 2) into a workspace of garbage equals the full
    backward bit for bit; pass 1 then 2 (D from the standalone pass) agrees within
    rounding."""
    B, T, H, Hkv, hd = 2, 300, 4, 2, 128
    q, k, v, do = inputs("bf16", B, T, T, H, Hkv, hd, 904, backward=True)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    kw = dict(H=H, Hkv=Hkv, causal=True)
    o, lse = A.attn_fwd(qd, kd, vd, **kw)
    n = A.attn_bwd_workspace_size(B, T, H)
    full = [t.clone() for t in A.attn_bwd(qd, kd, vd, o, dod, lse, **kw)]
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    dq4, _, _ = A.attn_bwd(qd, kd, vd, o, dod, lse, workspace=ws, phases=4, **kw)
    dq4 = dq4.clone()
    _, dk2, dv2 = A.attn_bwd(qd, kd, vd, o, dod, lse, workspace=ws, phases=2, **kw)
    torch.cuda.synchronize()
    assert torch.equal(dq4, full[0]) and torch.equal(dk2, full[1]) and torch.equal(dv2, full[2])
    ws.fill_(0xFF)
    A.attn_bwd(qd, kd, vd, o, dod, lse, workspace=ws, phases=1, **kw)
    _, dk1, dv1 = A.attn_bwd(qd, kd, vd, o, dod, lse, workspace=ws, phases=2, **kw)
    torch.cuda.synchronize()
    for a, b in ((dk1, full[1]), (dv1, full[2])):
        err = (a.float() - b.float()).norm() / b.float().norm()
        assert err < 1e-2, err


def test_guard_bands_untouched():
    """Outputs written inside larger buffers leave the surrounding canary bytes alone."""
    B, T, H, hd = 1, 130, 2, 64
    q, k, v, do = inputs("bf16", B, T, T, H, 1, hd, 903, backward=True)
    n = B * T * H * hd
    pad = 4096
    big = torch.full((n + 2 * pad,), 9.0, device="cuda", dtype=torch.bfloat16)
    o = big[pad:pad + n].view(B, T, H * hd)
    A.attn_fwd(q.cuda(), k.cuda(), v.cuda(), H=H, Hkv=1, causal=True, o=o)
    torch.cuda.synchronize()
    assert (big[:pad] == 9.0).all() and (big[pad + n:] == 9.0).all()


# In 16 bits hd 32 and 96 run on the tensor cores (padded), hd 256 too (the forward one
# query tile per work item, the backward in dV, dK and dQ passes); fp32 runs on the
# CUDA-core kernels.
@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("hd", [32, 96, 256])
def test_other_head_sizes_fwd_bwd(dt, hd):
    name = {"bf16": "bfloat16", "f32": "float32"}[dt]
    assert A.attn_kernel_family(name, hd) == (1 if dt != "f32" else 0)
    assert A.attn_kernel_family_bwd(name, hd) == (1 if dt != "f32" else 0)
    run_fwd_case(dt, 2, 150, 150, 4, 2, hd, causal=True, window=60, softcap=20.0, backward=True, seed=950 + hd)


HD256_FLAGS = [
    dict(causal=True),
    dict(causal=False),
    dict(causal=True, window=100, softcap=30.0),
    dict(causal=False, softcap=3.0, mask="batch"),
    dict(causal=True, mask="holes"),
    dict(causal=True, q_offset=90, window=200),
]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("flags", HD256_FLAGS, ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_fwd_hd256_tensor_core(dt, flags):
    """The hd 256 forward: several 64-key tiles and 128-row items, ragged tails, GQA."""
    Tq = 333
    run_fwd_case(dt, 2, Tq, Tq + flags.get("q_offset", 0), 4, 2, 256, seed=990, **flags)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("flags", HD256_FLAGS, ids=lambda f: "-".join("%s%s" % kv for kv in f.items()))
def test_bwd_hd256_tensor_core(dt, flags):
    """The hd 256 backward: two 64-row query tiles per GQA head and a ragged tail in
    each 128-key block of the dV / dK passes, several 64-key tiles per 128-row dQ block."""
    Tq = 333
    run_fwd_case(dt, 2, Tq, Tq + flags.get("q_offset", 0), 4, 2, 256, backward=True, seed=1990, **flags)


@pytest.mark.parametrize("case", [
    dict(B=1, Tq=5, Tk=70, H=2, Hkv=2, causal=False),                 # one query block, G = 1
    dict(B=2, Tq=64, Tk=65, H=3, Hkv=1, causal=True, q_offset=1),     # a key past one tile, G = 3
    dict(B=1, Tq=3, Tk=300, H=4, Hkv=2, causal=True, q_offset=297),   # decode-like rows
], ids=["tiny-g1", "tile-edge-g3", "decode-like"])
def test_bwd_hd256_edges(case):
    c = dict(case)
    B, Tq, Tk, H, Hkv = (c.pop(n) for n in ("B", "Tq", "Tk", "H", "Hkv"))
    run_fwd_case("bf16", B, Tq, Tk, H, Hkv, 256, backward=True, seed=1997, **c)


def test_bwd_hd256_many_blocks():
    # more key blocks and query blocks (3 x 8 x 3, 3 x 32 x 3) than SMs, group of four heads
    run_fwd_case("bf16", 3, 300, 300, 32, 8, 256, causal=True, backward=True, seed=1995)


def test_fwd_hd256_many_items_per_cta():
    # more 128-row items (3 x 32 x 3) than SMs: every CTA of the persistent kernel runs several
    run_fwd_case("bf16", 3, 300, 300, 32, 8, 256, causal=True, seed=995)


@pytest.mark.parametrize("hd", [32, 96])
def test_padded_head_sizes_multi_tile(hd):
    """Several query and key tiles, GQA and a ragged tail at the padded head sizes:
    a write past the head's columns would land in the next head's output."""
    run_fwd_case("bf16", 2, 700, 700, 8, 2, hd, causal=True, backward=True, seed=970 + hd)
    run_fwd_case("f16", 1, 333, 520, 6, 3, hd, causal=False, mask="batch", backward=True, seed=980 + hd)


@pytest.mark.parametrize("hd", [32, 96, 256])
def test_other_head_sizes_packed(hd):
    from attention_attn_fwd_08_gb300 import synth

    lens = [70, 0, 130, 1]
    cu = torch.tensor([0] + [int(x) for x in np.cumsum(lens)], dtype=torch.int32, device="cuda")
    tot = int(cu[-1])
    q = synth.normal((tot, 2 * hd), 960 + hd, "bf16")
    k = synth.normal((tot, hd), 961 + hd, "bf16")
    v = synth.normal((tot, hd), 962 + hd, "bf16")
    o, _ = A.attn_varlen_fwd(q.cuda(), k.cuda(), v.cuda(), cu, cu, 130, 130, H=2, Hkv=1, causal=True)
    torch.cuda.synchronize()
    ref, _ = oracle.varlen_fwd(f64(q), f64(k), f64(v), cu.tolist(), cu.tolist(), H=2, Hkv=1,
                               scale=1.0 / math.sqrt(hd), causal=True)
    assert np.abs(f64(o) - ref).max() <= 2e-2
