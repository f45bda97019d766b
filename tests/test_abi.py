"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments synchronously (before any CUDA call)."""
import ctypes
import os
import re

import pytest

import attention_attn_fwd_08_gb300 as A

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BAD = ctypes.c_void_p(0x1000)  # never dereferenced: every case fails validation first


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    L = A.lib()
    names = declared_symbols()
    assert {"attn_fwd", "attn_bwd", "attn_decode"} <= names
    for n in sorted(names):
        assert hasattr(L, n), n
    assert L.attn_abi_version() == 1


def test_status_strings():
    L = A.lib()
    for st in range(5):
        assert L.attn_status_string(st)
    assert b"invalid" in L.attn_status_string(1)


def fwd(**kw):
    args = dict(dt=2, q=BAD, k=BAD, v=BAD, o=BAD, lse=None, B=1, Tq=4, Tk=4, H=2, Hkv=1, hd=64, scale=0.125,
                causal=1, window=0, softcap=0.0, q_offset=0, mask=None, mstride=0, stream=None)
    args.update(kw)
    return A.lib().attn_fwd(*args.values())


@pytest.mark.parametrize("kw,expect", [
    (dict(H=3, Hkv=2), A.ERR_INVALID_ARG),         # Hkv must divide H
    (dict(Hkv=0), A.ERR_INVALID_ARG),
    (dict(hd=48), A.ERR_UNSUPPORTED),           # head sizes: 32, 64, 96, 128, 256
    (dict(hd=512), A.ERR_UNSUPPORTED),
    (dict(scale=0.0), A.ERR_INVALID_ARG),
    (dict(scale=float("nan")), A.ERR_INVALID_ARG),
    (dict(softcap=-1.0), A.ERR_INVALID_ARG),
    (dict(softcap=float("inf")), A.ERR_INVALID_ARG),
    (dict(window=-1), A.ERR_INVALID_ARG),
    (dict(q_offset=-1), A.ERR_INVALID_ARG),
    (dict(causal=2), A.ERR_INVALID_ARG),
    (dict(B=-1), A.ERR_INVALID_ARG),
    (dict(Tq=-1), A.ERR_INVALID_ARG),
    (dict(dt=7), A.ERR_INVALID_ARG),
    (dict(q=ctypes.c_void_p(0x1001)), A.ERR_INVALID_ARG),   # misaligned
    (dict(o=None), A.ERR_INVALID_ARG),                      # missing output
    (dict(mstride=-5), A.ERR_INVALID_ARG),
])
def test_fwd_rejects_bad_arguments(kw, expect):
    assert fwd(**kw) == expect


def test_empty_batch_or_queries_is_a_noop():
    assert fwd(B=0) == A.OK
    assert fwd(Tq=0) == A.OK


def test_bwd_and_decode_validation():
    L = A.lib()
    # bwd: workspace too small
    st = L.attn_bwd(2, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, 4, 1, 8, 8, 2, 1, 64, 0.125, 1, 0, 0.0,
                    0, None, 0, None)
    assert st == A.ERR_INVALID_ARG
    # decode: too many query rows per CTA group / too long a block
    st = L.attn_decode(2, BAD, BAD, BAD, BAD, None, BAD, 1 << 20, 1, 17, 64, 2, 1, 64, 0.125, 1, 0, 0.0, 47,
                       None, 0, None)
    assert st == A.ERR_UNSUPPORTED
    st = L.attn_decode(2, BAD, BAD, BAD, BAD, None, BAD, 1 << 20, 1, 16, 64, 8, 1, 64, 0.125, 1, 0, 0.0, 48,
                       None, 0, None)
    assert st == A.ERR_UNSUPPORTED
    # decode: workspace too small
    st = L.attn_decode(2, BAD, BAD, BAD, BAD, None, BAD, 16, 2, 4, 4096, 8, 2, 128, 0.1, 1, 0, 0.0, 4092,
                       None, 0, None)
    assert st == A.ERR_INVALID_ARG


def test_decode_len_validation():
    """Argument errors of the device-length decode come back before any launch."""
    L = A.lib()
    # NULL lengths
    st = L.attn_decode_len(2, BAD, BAD, BAD, BAD, None, BAD, 1 << 20, 2, 4, 256, 8, 2, 128, 0.1, 1, 0, 0.0, None,
                           None, 0, None)
    assert st == A.ERR_INVALID_ARG
    # lengths not 4-byte aligned
    st = L.attn_decode_len(2, BAD, BAD, BAD, BAD, None, BAD, 1 << 20, 2, 4, 256, 8, 2, 128, 0.1, 1, 0, 0.0, ctypes.c_void_p(0x1002),
                           None, 0, None)
    assert st == A.ERR_INVALID_ARG
    # fp32 has no split kernel
    st = L.attn_decode_len(0, BAD, BAD, BAD, BAD, None, BAD, 1 << 20, 2, 4, 256, 8, 2, 128, 0.1, 1, 0, 0.0, BAD,
                           None, 0, None)
    assert st == A.ERR_UNSUPPORTED
    # the 16-bit split kernel takes hd 64, 128, 256 (96 runs only through attn_fwd)
    st = L.attn_decode(2, BAD, BAD, BAD, BAD, None, BAD, 1 << 20, 2, 4, 256, 8, 2, 96, 0.1, 1, 0, 0.0, 252,
                       None, 0, None)
    assert st == A.ERR_UNSUPPORTED
    st = L.attn_decode(0, BAD, BAD, BAD, BAD, None, BAD, 1 << 20, 2, 4, 256, 8, 2, 48, 0.1, 1, 0, 0.0, 252,
                       None, 0, None)
    assert st == A.ERR_UNSUPPORTED
    st = L.attn_fwd(2, BAD, BAD, BAD, BAD, None, 2, 4, 256, 8, 2, 512, 0.1, 1, 0, 0.0, 0, None, 0, None)
    assert st == A.ERR_UNSUPPORTED
    # too long a query block
    st = L.attn_decode_len(2, BAD, BAD, BAD, BAD, None, BAD, 1 << 20, 2, 17, 256, 8, 2, 128, 0.1, 1, 0, 0.0, BAD,
                           None, 0, None)
    assert st == A.ERR_UNSUPPORTED
    # workspace too small for the capacity
    st = L.attn_decode_len(2, BAD, BAD, BAD, BAD, None, BAD, 16, 2, 4, 4096, 8, 2, 128, 0.1, 1, 0, 0.0, BAD,
                           None, 0, None)
    assert st == A.ERR_INVALID_ARG


def test_varlen_validation():
    """Argument errors of the packed-sequence calls come back before any launch."""
    L = A.lib()
    tail = [0.1, 1, 0, 0.0, None]
    # batch > 0 without cu_seqlens
    st = L.attn_varlen_fwd(2, BAD, BAD, BAD, BAD, None, None, None, 2, 64, 64, 100, 100, 8, 2, 128, *tail)
    assert st == A.ERR_INVALID_ARG
    # cu_seqlens not 4-byte aligned
    odd = ctypes.c_void_p(0x1002)
    st = L.attn_varlen_fwd(2, BAD, BAD, BAD, BAD, None, odd, BAD, 2, 64, 64, 100, 100, 8, 2, 128, *tail)
    assert st == A.ERR_INVALID_ARG
    # a bound above the packed row count
    st = L.attn_varlen_fwd(2, BAD, BAD, BAD, BAD, None, BAD, BAD, 2, 101, 64, 100, 100, 8, 2, 128, *tail)
    assert st == A.ERR_INVALID_ARG
    st = L.attn_varlen_fwd(2, BAD, BAD, BAD, BAD, None, BAD, BAD, 2, 64, 64, 100, -1, 8, 2, 128, *tail)
    assert st == A.ERR_INVALID_ARG
    # head dim, GQA divisibility, softcap
    st = L.attn_varlen_fwd(2, BAD, BAD, BAD, BAD, None, BAD, BAD, 2, 64, 64, 100, 100, 8, 2, 48, *tail)
    assert st == A.ERR_UNSUPPORTED
    st = L.attn_varlen_fwd(2, BAD, BAD, BAD, BAD, None, BAD, BAD, 2, 64, 64, 100, 100, 8, 3, 128, *tail)
    assert st == A.ERR_INVALID_ARG
    st = L.attn_varlen_fwd(2, BAD, BAD, BAD, BAD, None, BAD, BAD, 2, 64, 64, 100, 100, 8, 2, 128, 0.1, 1, 0, -1.0,
                           None)
    assert st == A.ERR_INVALID_ARG
    # nothing to do: no sequences, or no query rows
    assert L.attn_varlen_fwd(2, None, None, None, None, None, None, None, 0, 0, 0, 0, 0, 8, 2, 128, *tail) == A.OK
    assert L.attn_varlen_fwd(2, None, None, None, None, None, BAD, BAD, 3, 0, 5, 0, 5, 8, 2, 128, *tail) == A.OK
    # backward: workspace too small for batch x max_seqlen_q
    st = L.attn_varlen_bwd(2, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, 16, BAD, BAD, 2, 64, 64, 100, 100, 8,
                           2, 128, *tail)
    assert st == A.ERR_INVALID_ARG
    assert A.attn_bwd_workspace_size(2, 64, 8) > 16


def test_ex_validation():
    """Argument errors of the window/bias calls come back before any launch."""
    L = A.lib()
    args = [2, BAD, BAD, BAD, BAD, None, 2, 64, 64, 8, 2, 128, 0.1, 10, 0, 0.0, 0, None, 0]
    # bias not 4-byte aligned, negative bias stride
    assert L.attn_fwd_ex(*args, ctypes.c_void_p(0x1002), 0, 0, 64, 1, None) == A.ERR_INVALID_ARG
    assert L.attn_fwd_ex(*args, BAD, 0, 0, -64, 1, None) == A.ERR_INVALID_ARG
    # the usual shape rules
    bad_hd = [2, BAD, BAD, BAD, BAD, None, 2, 64, 64, 8, 2, 48, 0.1, 10, 0, 0.0, 0, None, 0]
    assert L.attn_fwd_ex(*bad_hd, None, 0, 0, 0, 0, None) == A.ERR_UNSUPPORTED
    st = L.attn_bwd_ex(2, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, 16, 2, 64, 64, 8, 2, 128, 0.1, 10, 0,
                       0.0, 0, None, 0, None, 0, 0, 0, 0, None)
    assert st == A.ERR_INVALID_ARG  # workspace too small
    # nothing to do
    zero = [2, None, None, None, None, None, 0, 64, 64, 8, 2, 128, 0.1, -1, -1, 0.0, 0, None, 0]
    assert L.attn_fwd_ex(*zero, None, 0, 0, 0, 0, None) == A.OK


def test_workspace_sizes():
    assert A.attn_bwd_workspace_size(4, 2048, 32) == 2 * 4 * 2048 * 32 * 4
    assert A.attn_bwd_workspace_size(1, 65, 2) == 2 * 1 * 128 * 2 * 4
    n = A.attn_decode_workspace_size(16, 4, 32768, 32, 8, 128)
    assert n > 0 and n % (16 * 32 * 4 * 130 * 4) == 0
    assert A.attn_decode_workspace_size(1, 1, 100, 3, 2, 128) == 0  # Hkv does not divide H
    assert A.attn_decode_workspace_size(2, 4, 1000, 8, 2, 256) > 0  # decode also takes hd 256


def test_kernel_family_is_reported():
    assert A.attn_kernel_family("float32", 64) == 0
    assert A.attn_kernel_family("bfloat16", 128) in (0, 1)


@pytest.mark.parametrize("B,Lq,Tk,H,Hkv", [
    (16, 1, 32768, 32, 8), (16, 4, 32768, 32, 8),   # the long-cache decode shapes
    (1, 1, 1, 1, 1), (1, 1, 63, 8, 8), (1, 1, 64, 8, 8), (1, 1, 65, 8, 8),
    (2, 16, 4096, 32, 8), (64, 16, 100000, 64, 1), (1, 3, 1 << 20, 8, 2), (3, 2, 777, 6, 3),
])
def test_decode_plan_partitions_the_cache(B, Lq, Tk, H, Hkv):
    """Host planning of the split-KV decode: the chunks tile [0, Tk) exactly, start on
    64-row boundaries, leave none empty, and the workspace holds one partial per
    (b, query head, row, chunk)."""
    splits, chunk = A.attn_decode_plan(B, Lq, Tk, H, Hkv)
    assert chunk > 0 and chunk % 64 == 0
    assert splits >= 1
    assert (splits - 1) * chunk < Tk <= splits * chunk  # every key in one chunk, the last chunk non-empty
    assert A.attn_decode_plan(B, Lq, Tk, H, Hkv) == (splits, chunk)  # deterministic
    for hd in (64, 128, 256):
        assert A.attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd) == B * H * Lq * splits * (hd + 2) * 4


def test_decode_plan_fills_the_gpu_on_long_caches():
    """A long cache with few (b, KV head) groups is split until the grid covers the
    152 SMs many times over; a large batch needs no split at all."""
    for B, Hkv in ((1, 1), (1, 8), (16, 8)):
        splits, chunk = A.attn_decode_plan(B, 1, 1 << 17, 8 * Hkv, Hkv)
        assert B * Hkv * splits >= 4 * 152, (B, Hkv, splits)
    splits, _ = A.attn_decode_plan(4096, 1, 1024, 32, 8)
    assert splits == 1
    # splitting stops at 64-row chunks
    assert A.attn_decode_plan(1, 1, 640, 1, 1) == (10, 64)


def test_decode_plan_validation():
    L = A.lib()
    one = ctypes.c_int(0)
    assert L.attn_decode_plan(1, 1, 16, 8, 2, None, ctypes.byref(one)) == A.ERR_INVALID_ARG
    for args in ((0, 1, 16, 8, 2), (1, 0, 16, 8, 2), (1, 1, -1, 8, 2), (1, 1, 16, 8, 3), (1, 1, 16, 0, 1)):
        with pytest.raises(A.AttnError):
            A.attn_decode_plan(*args)
    assert A.attn_decode_plan(2, 1, 0, 8, 2)[0] == 1  # an empty cache: one (empty) chunk
