"""Packed fused-QKV rows (attn_packed_qkv_fwd / _bwd) on the GPU against the fp64
oracle (oracle.packed_qkv_fwd / packed_qkv_bwd), through the C ABI: several packings
(long and one-row sequences, a single sequence), with and without the bidirectional
window, on the tensor-core kernels (16-bit hd 64 / 128) and the CUDA-core ones
(fp32, hd 96)."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_attn_fwd_08_gb300 as A
from attention_attn_fwd_08_gb300 import synth
from helpers import compare_grads, compare_o_lse, f64

pytestmark = pytest.mark.gpu

DT = {"bf16": "bfloat16", "f16": "float16", "f32": "float32"}


def bounds_of(lengths):
    L = int(sum(lengths))
    sb = np.zeros((L, 2), np.int32)
    s = 0
    for n in lengths:
        sb[s:s + n] = (s, s + n)
        s += n
    return torch.from_numpy(sb)


def run_packed(dt, lengths, H, hd, window, seed):
    sb = bounds_of(lengths)
    L = sb.shape[0]
    qkv = synth.normal((L, 3 * H * hd), seed, dt)
    do = synth.normal((L, H * hd), seed + 1, dt)
    scale = 1.0 / math.sqrt(hd)
    what = "%s L%d H%d hd%d window%d" % (dt, L, H, hd, window)
    o, lse = A.attn_packed_qkv_fwd(qkv.cuda(), sb.cuda(), H=H, window=window)
    dqkv = A.attn_packed_qkv_bwd(qkv.cuda(), do.cuda(), sb.cuda(), H=H, window=window)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    o_ref, lse_ref = oracle.packed_qkv_fwd(f64(qkv), sb.numpy(), H=H, scale=scale, window=window)
    compare_o_lse(o[None], lse[None], o_ref[None], lse_ref[None], dt, what)
    g_ref = oracle.packed_qkv_bwd(f64(qkv), f64(do), sb.numpy(), H=H, scale=scale, window=window)
    w = H * hd
    if max(lengths) == 1:
        # every row its own sequence: P = 1 and dS = 0, so dQ and dK vanish (a relative
        # error against the oracle's rounding-level zeros means nothing) and dV = dO.  The
        # 16-bit P of the forward leaves O within its rounding of v, and dQ, dK within
        # that of the gradients' scale, here the norm of dV.
        g = f64(dqkv)
        scale_g = np.linalg.norm(g_ref[:, 2 * w:])
        for name, c in (("dQ", 0), ("dK", 1)):
            e = np.linalg.norm(g[:, c * w:(c + 1) * w]) / scale_g
            assert e <= 5e-2, "%s: %s of one-row sequences %.3g of the gradient scale" % (what, name, e)
        assert np.abs(g[:, 2 * w:] - g_ref[:, 2 * w:]).max() <= 2e-2, what + ": dV of one-row sequences"
        return
    compare_grads((dqkv[:, :w], dqkv[:, w:2 * w], dqkv[:, 2 * w:]), (g_ref[:, :w], g_ref[:, w:2 * w], g_ref[:, 2 * w:]),
                  dt, what)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("window", [0, 9, 200])
def test_packed_qkv_tensor_cores(dt, hd, window):
    """Sequences longer and shorter than a tile, one-row ones, ragged tails."""
    assert A.attn_kernel_family(DT[dt], hd) == 1
    run_packed(dt, [300, 1, 129, 64, 2, 250], 2, hd, window, seed=2100 + hd + window)


@pytest.mark.parametrize("dt,hd", [("bf16", 64), ("f16", 128)])
def test_packed_qkv_tiles_far_apart(dt, hd):
    """A 256-row block whose first 128-row tile ends a long sequence and whose second lies
    in the next one: the two tiles' first key tiles are up to eight apart (their softmaxes
    must not take turns then), here with a window too."""
    for window in (0, 300):
        run_packed(dt, [600, 1000, 130, 900, 270], 2, hd, window, seed=2150 + hd + window)


@pytest.mark.parametrize("lengths", [[777], [1] * 40, [17, 300, 5, 500]], ids=["one-sequence", "one-row-each", "mixed"])
def test_packed_qkv_packings(lengths):
    run_packed("bf16", lengths, 4, 128, 0, seed=2200 + len(lengths))


@pytest.mark.parametrize("dt,hd", [("f32", 64), ("bf16", 96)])
def test_packed_qkv_cuda_cores(dt, hd):
    run_packed(dt, [70, 1, 33, 100], 2, hd, 16, seed=2300 + hd)


def test_packed_qkv_graph_replay_follows_bounds():
    """The launch shape depends on L only: a captured graph replays with a new packing."""
    L, H, hd = 300, 2, 64
    qkv = synth.normal((L, 3 * H * hd), 2400, "bf16").cuda()
    sb = bounds_of([100, 200]).cuda()
    o = torch.empty((L, H * hd), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((H, L), dtype=torch.float32, device="cuda")
    ws = torch.empty(A.attn_packed_qkv_workspace_size("bfloat16", L, H, hd), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        A.attn_packed_qkv_fwd(qkv, sb, H=H, o=o, lse=lse, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        A.attn_packed_qkv_fwd(qkv, sb, H=H, o=o, lse=lse, workspace=ws, stream=s)
    for lengths in ([100, 200], [1, 150, 149], [300]):
        sb.copy_(bounds_of(lengths).cuda())
        g.replay()
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle.packed_qkv_fwd(f64(qkv), bounds_of(lengths).numpy(), H=H, scale=1 / math.sqrt(hd))
        compare_o_lse(o[None], lse[None], o_ref[None], lse_ref[None], "bf16", "graph %s" % (lengths,))


def test_packed_qkv_rejects_bad_arguments():
    qkv = torch.zeros((8, 3 * 2 * 64), dtype=torch.bfloat16, device="cuda")
    sb = bounds_of([8]).cuda()
    with pytest.raises(ValueError):
        A.attn_packed_qkv_fwd(qkv, sb.to(torch.int64), H=2)
    with pytest.raises(ValueError):
        A.attn_packed_qkv_fwd(qkv, sb[:4], H=2)
    with pytest.raises(A.AttnError):
        A.attn_packed_qkv_fwd(qkv, sb, H=2, window=-1)


@pytest.mark.parametrize("window", [0, 128])
def test_packed_qkv_full_size(window):
    """The benchmark's packing (16 sequences of U{128..1024} rows, H=12 hd=64 bf16),
    forward and backward in one call each as timed; sequences are independent, so the
    shortest, a middle and the longest one are checked against the oracle run on that
    sequence's rows alone."""
    w = synth.WORKLOADS["packed_qkv"]
    pi = synth.make_packed_qkv_inputs(w)
    qkv, do, sb = pi["qkv"], pi["do"], pi["seq_bounds"]
    o, lse = A.attn_packed_qkv_fwd(qkv.cuda(), sb.cuda(), H=w.H, window=window)
    dqkv = A.attn_packed_qkv_bwd(qkv.cuda(), do.cuda(), sb.cuda(), H=w.H, window=window)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    o, lse, dqkv = o.cpu(), lse.cpu(), dqkv.cpu()
    lens = pi["lengths"].tolist()
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    order = np.argsort(lens, kind="stable")
    nw = w.H * w.hd
    for s in sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])}):
        a, n = int(starts[s]), int(lens[s])
        rows = slice(a, a + n)
        sub = bounds_of([n]).numpy()
        what = "packed_qkv window %d, sequence %d (%d rows)" % (window, s, n)
        o_ref, lse_ref = oracle.packed_qkv_fwd(f64(qkv[rows]), sub, H=w.H, scale=w.scale, window=window)
        compare_o_lse(o[rows][None], lse[:, rows][None], o_ref[None], lse_ref[None], "bf16", what)
        g_ref = oracle.packed_qkv_bwd(f64(qkv[rows]), f64(do[rows]), sub, H=w.H, scale=w.scale, window=window)
        g = dqkv[rows]
        compare_grads((g[:, :nw], g[:, nw:2 * nw], g[:, 2 * nw:]),
                      (g_ref[:, :nw], g_ref[:, nw:2 * nw], g_ref[:, 2 * nw:]), "bf16", what)


def test_packed_qkv_past_the_block_order():
    """More than 2048 blocks of 128 rows (262 145 rows): the kernels keep their plain item
    order (no heaviest-first pass) and large row indices; three sequences are checked
    against the oracle, forward and backward."""
    H, hd, n = 1, 64, 256
    lengths = [1024] * n
    lengths[-1] += 1
    sb = bounds_of(lengths)
    L = sb.shape[0]
    assert (L + 127) // 128 > 2048
    qkv = synth.normal((L, 3 * H * hd), 2500, "bf16")
    do = synth.normal((L, H * hd), 2501, "bf16")
    o, lse = A.attn_packed_qkv_fwd(qkv.cuda(), sb.cuda(), H=H)
    dqkv = A.attn_packed_qkv_bwd(qkv.cuda(), do.cuda(), sb.cuda(), H=H)
    torch.cuda.synchronize()
    st, word = A.attn_get_device_status()
    assert st == A.OK, "device status word %#x" % word
    o, lse, dqkv = o.cpu(), lse.cpu(), dqkv.cpu()
    for s in (0, n // 2, n - 1):
        a = 1024 * s
        rows = slice(a, a + lengths[s])
        sub = bounds_of([lengths[s]]).numpy()
        what = "packed_qkv L%d, sequence %d" % (L, s)
        o_ref, lse_ref = oracle.packed_qkv_fwd(f64(qkv[rows]), sub, H=H, scale=1 / math.sqrt(hd))
        compare_o_lse(o[rows][None], lse[:, rows][None], o_ref[None], lse_ref[None], "bf16", what)
        g_ref = oracle.packed_qkv_bwd(f64(qkv[rows]), f64(do[rows]), sub, H=H, scale=1 / math.sqrt(hd))
        g = dqkv[rows]
        compare_grads((g[:, :hd], g[:, hd:2 * hd], g[:, 2 * hd:]), (g_ref[:, :hd], g_ref[:, hd:2 * hd], g_ref[:, 2 * hd:]),
                      "bf16", what)
