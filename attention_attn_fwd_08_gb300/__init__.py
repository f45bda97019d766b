"""GB300 fused attention: a thin ctypes binding over libattn_gb300.so.

The functions here only marshal arguments: they check tensor shapes, let
PyTorch allocate outputs and scratch, and call the C ABI of include/attn.h
with raw device pointers and the current CUDA stream.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback, and a missing or unloadable library raises.

    o, lse = attn_fwd(q, k, v, H=32, Hkv=8, causal=True)
    dq, dk, dv = attn_bwd(q, k, v, o, do, lse, H=32, Hkv=8, causal=True)
    o, lse = attn_decode(q, k_cache, v_cache, H=32, Hkv=8, causal=True, q_offset=Tk - Lq)

Layouts: q/o/do/dq [B, Tq, H*hd]; k/v/dk/dv [B, Tk, Hkv*hd]; lse [B, H, Tq] fp32;
key_mask fp32 [Tk] (shared) or [B, Tk].
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = ["attn_fwd", "attn_bwd", "attn_decode", "attn_decode_len", "attn_varlen_fwd", "attn_varlen_bwd", "attn_fwd_ex", "attn_bwd_ex", "attn_rope", "attn_bwd_workspace_size", "attn_decode_workspace_size", "attn_decode_plan",
           "attn_get_device_status", "attn_selftest_bounded_wait", "attn_kernel_family", "attn_kernel_family_bwd", "attn_fwd_rope", "attn_bwd_rope", "attn_fwd_rope_workspace_size", "attn_bwd_rope_workspace_size", "attn_launch_count", "attn_packed_qkv_fwd", "attn_packed_qkv_bwd", "attn_packed_qkv_workspace_size", "AttnError", "lib",
           "library_path"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
_DT = {"float32": 0, "float16": 1, "bfloat16": 2}


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, _status_string(status), status))


def library_path() -> str:
    return os.path.join(_HERE, "libattn_gb300.so")


def lib():
    """The loaded C library (built in-tree on first use if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build as _build

        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i, f, ll, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_size_t
        tail = [i, i, i, i, i, i, f, i, i, f, i, vp, ll, vp]
        L.attn_fwd.argtypes = [i, vp, vp, vp, vp, vp] + tail
        L.attn_fwd.restype = i
        L.attn_bwd_workspace_size.argtypes = [i, i, i]
        L.attn_bwd_workspace_size.restype = sz
        L.attn_bwd.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz] + tail
        L.attn_bwd.restype = i
        L.attn_bwd_phases.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz] + tail + [i]
        L.attn_bwd_phases.restype = i
        L.attn_launch_count.argtypes = []
        L.attn_launch_count.restype = ctypes.c_ulonglong
        L.attn_decode_workspace_size.argtypes = [i, i, i, i, i, i]
        L.attn_decode_workspace_size.restype = sz
        L.attn_decode_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        L.attn_decode_plan.restype = i
        L.attn_decode.argtypes = [i, vp, vp, vp, vp, vp, vp, sz] + tail
        L.attn_decode.restype = i
        L.attn_decode_len.argtypes = [i, vp, vp, vp, vp, vp, vp, sz] + [i] * 6 + [f, i, i, f, vp, vp, ll, vp]
        L.attn_decode_len.restype = i
        tail_ex = [i, i, i, i, i, i, f, i, i, f, i, vp, ll, vp, ll, ll, ll, ll, vp]
        L.attn_fwd_ex.argtypes = [i, vp, vp, vp, vp, vp] + tail_ex
        L.attn_fwd_ex.restype = i
        L.attn_bwd_ex.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz] + tail_ex
        L.attn_bwd_ex.restype = i
        L.attn_rope.argtypes = [i, vp, i, i, i, i, i, f, vp]
        L.attn_rope.restype = i
        L.attn_varlen_fwd.argtypes = [i] + [vp] * 7 + [i] * 8 + [f, i, i, f, vp]
        L.attn_varlen_fwd.restype = i
        L.attn_varlen_bwd.argtypes = [i] + [vp] * 10 + [sz, vp, vp] + [i] * 8 + [f, i, i, f, vp]
        L.attn_varlen_bwd.restype = i
        L.attn_packed_qkv_workspace_size.argtypes = [i, i, i, i, i]
        L.attn_packed_qkv_workspace_size.restype = sz
        L.attn_packed_qkv_fwd.argtypes = [i, vp, vp, vp, vp, vp, sz, i, i, i, f, i, vp]
        L.attn_packed_qkv_fwd.restype = i
        L.attn_packed_qkv_bwd.argtypes = [i, vp, vp, vp, vp, vp, sz, i, i, i, f, i, vp]
        L.attn_packed_qkv_bwd.restype = i
        L.attn_status_string.argtypes = [i]
        L.attn_status_string.restype = ctypes.c_char_p
        L.attn_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
        L.attn_get_device_status.restype = i
        L.attn_selftest_bounded_wait.argtypes = [ctypes.c_uint, vp]
        L.attn_selftest_bounded_wait.restype = i
        L.attn_kernel_family.argtypes = [i, i]
        L.attn_kernel_family.restype = i
        L.attn_kernel_family_bwd.argtypes = [i, i]
        L.attn_kernel_family_bwd.restype = i
        L.attn_fwd_rope_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
        L.attn_fwd_rope_workspace_size.restype = sz
        L.attn_fwd_rope.argtypes = [i, vp, vp, vp, vp, vp, vp, sz] + [i] * 6 + [f, i, i, f, i, vp, ll, i, f, vp]
        L.attn_fwd_rope.restype = i
        L.attn_bwd_rope_workspace_size.argtypes = [i, i, i, i, i, i, i]
        L.attn_bwd_rope_workspace_size.restype = sz
        L.attn_bwd_rope.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz] + [i] * 6 + [f, i, i, f, i, vp, ll,
                                                                                           i, f, vp]
        L.attn_bwd_rope.restype = i
        L.attn_abi_version.argtypes = []
        L.attn_abi_version.restype = i
        _lib = L
        return L


def _status_string(st: int) -> str:
    try:
        return lib().attn_status_string(int(st)).decode()
    except Exception:  # the library itself failed to load
        return "status %d" % st


def _check(st: int, what: str):
    if st != OK:
        raise AttnError(st, what)


def _torch():
    import torch

    return torch


def _dt(t) -> int:
    name = str(t.dtype).replace("torch.", "")
    if name not in _DT:
        raise TypeError("unsupported dtype %s" % t.dtype)
    return _DT[name]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dims(q, k, H, Hkv):
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q must be [B,Tq,H*hd] and k/v [B,Tk,Hkv*hd]")
    B, Tq, qc = q.shape
    Bk, Tk, kc = k.shape
    if Bk != B or qc % H or kc % Hkv or qc // H != kc // Hkv:
        raise ValueError("inconsistent shapes: q %s, k %s, H=%d, Hkv=%d" % (tuple(q.shape), tuple(k.shape), H, Hkv))
    return B, Tq, Tk, qc // H


def _mask(key_mask, B, Tk):
    if key_mask is None:
        return None, 0
    if key_mask.dtype != _torch().float32 or not key_mask.is_contiguous():
        raise ValueError("key_mask must be a contiguous fp32 tensor")
    if key_mask.dim() == 1:
        if key_mask.shape[0] != Tk:
            raise ValueError("key_mask must have Tk entries")
        return key_mask, 0
    if tuple(key_mask.shape) != (B, Tk):
        raise ValueError("key_mask must be [Tk] or [B,Tk]")
    return key_mask, Tk


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _placed(q, like_q=(), like_k=(), k=None, f32=(), device=()):
    """Checks, before any pointer reaches the library, what it cannot check itself:
    every tensor in like_q / like_k is on q's device with q's dtype and the shape of
    q / k; every (name, tensor, shape) in f32 is an fp32 tensor of that shape on q's
    device; every tensor in device is on q's device; and that device is a GPU (a host
    pointer would reach the kernels as a device address).  Entries may be None."""
    for group, ref in ((like_q, q), (like_k, k)):
        for name, t in group:
            if t is None:
                continue
            if t.device != q.device or t.dtype != q.dtype:
                raise ValueError("%s must be a %s tensor on %s (got %s on %s)" % (name, q.dtype, q.device, t.dtype,
                                                                                t.device))
            if tuple(t.shape) != tuple(ref.shape):
                raise ValueError("%s must have shape %s (got %s)" % (name, tuple(ref.shape), tuple(t.shape)))
    for name, t, shape in f32:
        if t is None:
            continue
        if t.device != q.device or t.dtype != _torch().float32 or tuple(t.shape) != tuple(shape):
            raise ValueError("%s must be an fp32 tensor of shape %s on %s" % (name, tuple(shape), q.device))
    for name, t in device:
        if t is not None and t.device != q.device:
            raise ValueError("%s must be on %s (got %s)" % (name, q.device, t.device))
    if q.device.type != "cuda":
        raise ValueError("the library takes CUDA tensors; q is on %s" % q.device)


def attn_fwd(q, k, v, *, H, Hkv, scale=None, causal=False, window=0, softcap=0.0, q_offset=0, key_mask=None,
             o=None, lse=None, want_lse=True, stream=None):
    """Forward attention; returns (o, lse).  lse is None when want_lse is False."""
    torch = _torch()
    _contig(q, k, v, o, lse)
    B, Tq, Tk, hd = _dims(q, k, H, Hkv)
    _placed(q, like_q=[("o", o)], like_k=[("k", k), ("v", v)], k=k, f32=[("lse", lse, (B, H, Tq))],
            device=[("key_mask", key_mask)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    m, ms = _mask(key_mask, B, Tk)
    st = lib().attn_fwd(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Tq, Tk, H, Hkv, hd,
                        float(scale), int(bool(causal)), int(window), float(softcap), int(q_offset), _ptr(m),
                        int(ms), _stream(stream))
    _check(st, "attn_fwd")
    return o, lse


def attn_bwd_workspace_size(B, Tq, H) -> int:
    return int(lib().attn_bwd_workspace_size(B, Tq, H))


def attn_bwd(q, k, v, o, do, lse, *, H, Hkv, scale=None, causal=False, window=0, softcap=0.0, q_offset=0,
             key_mask=None, dq=None, dk=None, dv=None, workspace=None, stream=None, phases=7):
    """Backward attention; returns (dq, dk, dv), overwritten.

    phases selects passes (1 = D = rowsum(dO*O), 2 = dK/dV, 4 = dQ, which forms D
    itself); pass 2 alone reads the D that an earlier pass 1 or 4 left in
    `workspace`, so pass the same workspace."""
    torch = _torch()
    _contig(q, k, v, o, do, lse, dq, dk, dv)
    B, Tq, Tk, hd = _dims(q, k, H, Hkv)
    _placed(q, like_q=[("o", o), ("do", do), ("dq", dq)], like_k=[("k", k), ("v", v), ("dk", dk), ("dv", dv)], k=k,
            f32=[("lse", lse, (B, H, Tq))], device=[("key_mask", key_mask), ("workspace", workspace)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = attn_bwd_workspace_size(B, Tq, H)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    m, ms = _mask(key_mask, B, Tk)
    st = lib().attn_bwd_phases(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                               _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               B, Tq, Tk, H, Hkv, hd, float(scale), int(bool(causal)), int(window), float(softcap),
                               int(q_offset), _ptr(m), int(ms), _stream(stream), int(phases))
    _check(st, "attn_bwd")
    return dq, dk, dv


def attn_fwd_rope_workspace_size(dtype, B, Tq, Tk, H, Hkv, hd, q_offset=0) -> int:
    return int(lib().attn_fwd_rope_workspace_size(_DT[dtype], B, Tq, Tk, H, Hkv, hd, int(q_offset)))


def attn_fwd_rope(q, k, v, *, H, Hkv, scale=None, causal=False, window=0, softcap=0.0, q_offset=0, key_mask=None,
                  rope_pos=0, rope_theta=10000.0, o=None, lse=None, want_lse=True, workspace=None, stream=None):
    """Forward attention on the rotary-embedded q and k (q and k are passed unrotated and
    left unchanged): query row i turns at position rope_pos + q_offset + i, key j at
    rope_pos + j.  Returns (o, lse)."""
    torch = _torch()
    _contig(q, k, v, o, lse)
    B, Tq, Tk, hd = _dims(q, k, H, Hkv)
    _placed(q, like_q=[("o", o)], like_k=[("k", k), ("v", v)], k=k, f32=[("lse", lse, (B, H, Tq))],
            device=[("key_mask", key_mask), ("workspace", workspace)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    name = str(q.dtype).split(".")[-1]
    if workspace is None:
        nbytes = attn_fwd_rope_workspace_size(name, B, Tq, Tk, H, Hkv, hd, q_offset)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    m, ms = _mask(key_mask, B, Tk)
    st = lib().attn_fwd_rope(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), B, Tq, Tk, H, Hkv, hd, float(scale),
                             int(bool(causal)), int(window), float(softcap), int(q_offset), _ptr(m), int(ms),
                             int(rope_pos), float(rope_theta), _stream(stream))
    _check(st, "attn_fwd_rope")
    return o, lse


def attn_bwd_rope_workspace_size(dtype, B, Tq, Tk, H, Hkv, hd) -> int:
    return int(lib().attn_bwd_rope_workspace_size(_DT[dtype], B, Tq, Tk, H, Hkv, hd))


def attn_bwd_rope(q, k, v, o, do, lse, *, H, Hkv, scale=None, causal=False, window=0, softcap=0.0, q_offset=0,
                  key_mask=None, rope_pos=0, rope_theta=10000.0, dq=None, dk=None, dv=None, workspace=None,
                  stream=None):
    """Backward of attn_fwd_rope (same arguments; o and lse from that call): returns
    (dq, dk, dv), the gradients of the unrotated q and k, overwritten."""
    torch = _torch()
    _contig(q, k, v, o, do, lse, dq, dk, dv)
    B, Tq, Tk, hd = _dims(q, k, H, Hkv)
    _placed(q, like_q=[("o", o), ("do", do), ("dq", dq)], like_k=[("k", k), ("v", v), ("dk", dk), ("dv", dv)], k=k,
            f32=[("lse", lse, (B, H, Tq))], device=[("key_mask", key_mask), ("workspace", workspace)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    name = str(q.dtype).split(".")[-1]
    if workspace is None:
        nbytes = attn_bwd_rope_workspace_size(name, B, Tq, Tk, H, Hkv, hd)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    m, ms = _mask(key_mask, B, Tk)
    st = lib().attn_bwd_rope(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(), B, Tq, Tk, H,
                             Hkv, hd, float(scale), int(bool(causal)), int(window), float(softcap), int(q_offset),
                             _ptr(m), int(ms), int(rope_pos), float(rope_theta), _stream(stream))
    _check(st, "attn_bwd_rope")
    return dq, dk, dv


def attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd) -> int:
    return int(lib().attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd))


def attn_decode_plan(B, Lq, Tk, H, Hkv):
    """(splits, chunk): the decode calls' key split for this shape (host only)."""
    splits, chunk = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().attn_decode_plan(B, Lq, Tk, H, Hkv, ctypes.byref(splits), ctypes.byref(chunk)), "attn_decode_plan")
    return splits.value, chunk.value


def attn_decode(q, k, v, *, H, Hkv, scale=None, causal=True, window=0, softcap=0.0, q_offset=None, key_mask=None,
                o=None, lse=None, want_lse=True, workspace=None, stream=None):
    """Split-KV decode of an Lq-row block; q_offset defaults to Tk - Lq. Returns (o, lse)."""
    torch = _torch()
    _contig(q, k, v, o, lse)
    B, Lq, Tk, hd = _dims(q, k, H, Hkv)
    _placed(q, like_q=[("o", o)], like_k=[("k", k), ("v", v)], k=k, f32=[("lse", lse, (B, H, Lq))],
            device=[("key_mask", key_mask), ("workspace", workspace)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    q_offset = Tk - Lq if q_offset is None else q_offset
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    nbytes = attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    m, ms = _mask(key_mask, B, Tk)
    st = lib().attn_decode(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), B, Lq, Tk, H, Hkv, hd, float(scale),
                           int(bool(causal)), int(window), float(softcap), int(q_offset), _ptr(m), int(ms),
                           _stream(stream))
    _check(st, "attn_decode")
    return o, lse


def attn_decode_len(q, k, v, lengths, *, H, Hkv, scale=None, causal=True, window=0, softcap=0.0, key_mask=None,
                    o=None, lse=None, want_lse=True, workspace=None, stream=None):
    """Split-KV decode over a cache of capacity k.shape[1] whose per-sequence valid
    length is read on the device from `lengths` (int32 [B]); the Lq query rows of
    sequence b sit at positions lengths[b] - Lq .. lengths[b] - 1.  Returns (o, lse).
    The launch depends on the capacity only, so it can be captured in a CUDA graph
    and replayed after `lengths` changes."""
    torch = _torch()
    _contig(q, k, v, o, lse, lengths)
    B, Lq, Tk, hd = _dims(q, k, H, Hkv)
    _placed(q, like_q=[("o", o)], like_k=[("k", k), ("v", v)], k=k, f32=[("lse", lse, (B, H, Lq))],
            device=[("key_mask", key_mask), ("workspace", workspace), ("lengths", lengths)])
    if lengths.dtype != torch.int32 or lengths.numel() != B:
        raise ValueError("lengths must be int32 with one entry per batch")
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    nbytes = attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    m, ms = _mask(key_mask, B, Tk)
    st = lib().attn_decode_len(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), B, Lq, Tk, H, Hkv, hd, float(scale),
                               int(bool(causal)), int(window), float(softcap), _ptr(lengths), _ptr(m), int(ms),
                               _stream(stream))
    _check(st, "attn_decode_len")
    return o, lse


def _bias(bias, B, H, Tq, Tk):
    """(tensor or None, 4 strides in elements) of a bias broadcastable to [B, H, Tq, Tk]."""
    if bias is None:
        return None, (0, 0, 0, 0)
    torch = _torch()
    if bias.dtype != torch.float32 or bias.dim() != 4:
        raise ValueError("bias must be a 4-D fp32 tensor [B|1, H|1, Tq|1, Tk|1]")
    st = []
    for dim, n, s in zip(bias.shape, (B, H, Tq, Tk), bias.stride()):
        if dim not in (1, n):
            raise ValueError("bias shape %s does not broadcast to %s" % (tuple(bias.shape), (B, H, Tq, Tk)))
        st.append(0 if dim == 1 else s)
    return bias, tuple(st)


def attn_fwd_ex(q, k, v, *, H, Hkv, scale=None, window_left=-1, window_right=-1, softcap=0.0, q_offset=0,
                key_mask=None, bias=None, o=None, lse=None, want_lse=True, stream=None):
    """Forward with the two-sided window [p - window_left, p + window_right] (negative:
    unbounded) and an optional fp32 additive bias broadcastable to [B, H, Tq, Tk]."""
    torch = _torch()
    _contig(q, k, v, o, lse)
    B, Tq, Tk, hd = _dims(q, k, H, Hkv)
    _placed(q, like_q=[("o", o)], like_k=[("k", k), ("v", v)], k=k, f32=[("lse", lse, (B, H, Tq))],
            device=[("key_mask", key_mask), ("bias", bias)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    m, ms = _mask(key_mask, B, Tk)
    bt, bs = _bias(bias, B, H, Tq, Tk)
    st = lib().attn_fwd_ex(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Tq, Tk, H, Hkv, hd, float(scale),
                           int(window_left), int(window_right), float(softcap), int(q_offset), _ptr(m), int(ms),
                           _ptr(bt), *bs, _stream(stream))
    _check(st, "attn_fwd_ex")
    return o, lse


def attn_bwd_ex(q, k, v, o, do, lse, *, H, Hkv, scale=None, window_left=-1, window_right=-1, softcap=0.0,
                q_offset=0, key_mask=None, bias=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of attn_fwd_ex (same window and bias); returns (dq, dk, dv), overwritten."""
    torch = _torch()
    _contig(q, k, v, o, do, lse, dq, dk, dv)
    B, Tq, Tk, hd = _dims(q, k, H, Hkv)
    _placed(q, like_q=[("o", o), ("do", do), ("dq", dq)], like_k=[("k", k), ("v", v), ("dk", dk), ("dv", dv)], k=k,
            f32=[("lse", lse, (B, H, Tq))], device=[("key_mask", key_mask), ("bias", bias), ("workspace", workspace)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = attn_bwd_workspace_size(B, Tq, H)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    m, ms = _mask(key_mask, B, Tk)
    bt, bs = _bias(bias, B, H, Tq, Tk)
    st = lib().attn_bwd_ex(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                           _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(), B, Tq, Tk, H, Hkv,
                           hd, float(scale), int(window_left), int(window_right), float(softcap), int(q_offset),
                           _ptr(m), int(ms), _ptr(bt), *bs, _stream(stream))
    _check(st, "attn_bwd_ex")
    return dq, dk, dv


def attn_rope(x, *, H, pos=0, theta=10000.0, stream=None):
    """Rotate-half rotary embedding of x [B, T, H*hd] in place (every head vector of
    token s at position pos + s); returns x."""
    _contig(x)
    _placed(x)
    if x.dim() != 3 or x.shape[2] % H:
        raise ValueError("x must be [B, T, H*hd]")
    B, T, C = x.shape
    st = lib().attn_rope(_dt(x), _ptr(x), B, T, H, C // H, int(pos), float(theta), _stream(stream))
    _check(st, "attn_rope")
    return x


def _varlen_dims(q, k, cu_q, cu_k, H, Hkv):
    torch = _torch()
    if q.dim() != 2 or k.dim() != 2:
        raise ValueError("packed q must be [total_q, H*hd] and k/v [total_k, Hkv*hd]")
    if q.shape[1] % H or k.shape[1] % Hkv or q.shape[1] // H != k.shape[1] // Hkv:
        raise ValueError("inconsistent shapes: q %s, k %s, H=%d, Hkv=%d" % (tuple(q.shape), tuple(k.shape), H, Hkv))
    for c in (cu_q, cu_k):
        if c.dtype != torch.int32 or c.dim() != 1 or not c.is_contiguous():
            raise ValueError("cu_seqlens must be contiguous int32 [batch+1]")
    if cu_q.numel() != cu_k.numel() or cu_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have batch+1 entries")
    return cu_q.numel() - 1, q.shape[0], k.shape[0], q.shape[1] // H


def attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *, H, Hkv, scale=None,
                    causal=False, window=0, softcap=0.0, o=None, lse=None, want_lse=True, stream=None):
    """Packed variable-length forward: sequence b owns rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
    of q/o and cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 of k/v (int32 device prefix sums); no
    attention across sequences.  Returns (o, lse), lse [batch, H, max_seqlen_q].  Rows of o
    outside every sequence are left as they were."""
    torch = _torch()
    _contig(q, k, v, o, lse)
    batch, total_q, total_k, hd = _varlen_dims(q, k, cu_seqlens_q, cu_seqlens_k, H, Hkv)
    _placed(q, like_q=[("o", o)], like_k=[("k", k), ("v", v)], k=k, f32=[("lse", lse, (batch, H, max_seqlen_q))],
            device=[("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((batch, H, max_seqlen_q), dtype=torch.float32, device=q.device)
    st = lib().attn_varlen_fwd(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                               _ptr(cu_seqlens_k), batch, int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, H,
                               Hkv, hd, float(scale), int(bool(causal)), int(window), float(softcap), _stream(stream))
    _check(st, "attn_varlen_fwd")
    return o, lse


def attn_varlen_bwd(q, k, v, o, do, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *, H, Hkv,
                    scale=None, causal=False, window=0, softcap=0.0, dq=None, dk=None, dv=None, workspace=None,
                    stream=None):
    """Backward of attn_varlen_fwd; returns (dq, dk, dv), overwritten on every sequence's rows."""
    torch = _torch()
    _contig(q, k, v, o, do, lse, dq, dk, dv)
    batch, total_q, total_k, hd = _varlen_dims(q, k, cu_seqlens_q, cu_seqlens_k, H, Hkv)
    _placed(q, like_q=[("o", o), ("do", do), ("dq", dq)], like_k=[("k", k), ("v", v), ("dk", dk), ("dv", dv)], k=k,
            f32=[("lse", lse, (batch, H, max_seqlen_q))],
            device=[("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k), ("workspace", workspace)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = attn_bwd_workspace_size(batch, int(max_seqlen_q), H)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = lib().attn_varlen_bwd(_dt(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, int(max_seqlen_q), int(max_seqlen_k),
                               total_q, total_k, H, Hkv, hd, float(scale), int(bool(causal)), int(window),
                               float(softcap), _stream(stream))
    _check(st, "attn_varlen_bwd")
    return dq, dk, dv


def attn_get_device_status(stream=None):
    """(status, detail word); reads and clears the device status word."""
    w = ctypes.c_uint(0)
    st = lib().attn_get_device_status(_stream(stream), ctypes.byref(w))
    return int(st), int(w.value)


def attn_selftest_bounded_wait(timeout_us: int, stream=None):
    _check(lib().attn_selftest_bounded_wait(int(timeout_us), _stream(stream)), "attn_selftest_bounded_wait")


def attn_launch_count() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib().attn_launch_count())


def attn_kernel_family(dtype: str, hd: int) -> int:
    """1 when attn_fwd runs (dtype, hd) on the tensor cores, 0 on the CUDA-core kernels."""
    return int(lib().attn_kernel_family(_DT[dtype], int(hd)))


def attn_kernel_family_bwd(dtype: str, hd: int) -> int:
    """1 when attn_bwd runs (dtype, hd) on the tensor cores, 0 on the CUDA-core kernels."""
    return int(lib().attn_kernel_family_bwd(_DT[dtype], int(hd)))


# ------------------------------------------------------------ packed fused-QKV rows
def _packed_dims(qkv, seq_bounds, H):
    torch = _torch()
    if qkv.dim() != 2 or qkv.shape[1] % (3 * H):
        raise ValueError("qkv must be [L, 3*H*hd]")
    L = int(qkv.shape[0])
    if seq_bounds.dtype != torch.int32 or tuple(seq_bounds.shape) != (L, 2) or not seq_bounds.is_contiguous():
        raise ValueError("seq_bounds must be a contiguous int32 tensor of shape [L, 2]")
    return L, int(qkv.shape[1]) // (3 * H)


def attn_packed_qkv_workspace_size(dtype: str, L: int, H: int, hd: int, backward: bool = False) -> int:
    """Workspace bytes attn_packed_qkv_fwd (or, with backward, attn_packed_qkv_bwd) needs."""
    return int(lib().attn_packed_qkv_workspace_size(_DT[dtype], int(L), int(H), int(hd), int(bool(backward))))


def attn_packed_qkv_fwd(qkv, seq_bounds, *, H, scale=None, window=0, o=None, lse=None, want_lse=True, workspace=None,
                        stream=None):
    """Packed bidirectional self-attention off a fused QKV projection: qkv [L, 3*H*hd] rows
    [q heads | k heads | v heads]; row r attends the keys of its own sequence, rows
    seq_bounds[r, 0] .. seq_bounds[r, 1]-1 (int32 [L, 2] on the device), within
    |r - j| <= window // 2 when window > 0.  Returns (o [L, H*hd], lse [H, L])."""
    torch = _torch()
    _contig(qkv, seq_bounds, o, lse)
    L, hd = _packed_dims(qkv, seq_bounds, H)
    if o is not None and (o.device != qkv.device or o.dtype != qkv.dtype or tuple(o.shape) != (L, H * hd)):
        raise ValueError("o must be a %s tensor of shape %s on %s" % (qkv.dtype, (L, H * hd), qkv.device))
    _placed(qkv, f32=[("lse", lse, (H, L))], device=[("seq_bounds", seq_bounds), ("workspace", workspace)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    o = torch.empty((L, H * hd), dtype=qkv.dtype, device=qkv.device) if o is None else o
    if lse is None and want_lse:
        lse = torch.empty((H, L), dtype=torch.float32, device=qkv.device)
    nbytes = lib().attn_packed_qkv_workspace_size(_dt(qkv), L, H, hd, 0)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=qkv.device)
    st = lib().attn_packed_qkv_fwd(_dt(qkv), _ptr(qkv), _ptr(seq_bounds), _ptr(o), _ptr(lse), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), L, H, hd, float(scale), int(window),
                                   _stream(stream))
    _check(st, "attn_packed_qkv_fwd")
    return o, lse


def attn_packed_qkv_bwd(qkv, do, seq_bounds, *, H, scale=None, window=0, dqkv=None, workspace=None, stream=None):
    """Backward of attn_packed_qkv_fwd from do [L, H*hd]: returns dqkv [L, 3*H*hd] (rows
    [dq | dk | dv]), overwritten; O and LSE are formed again from qkv."""
    torch = _torch()
    _contig(qkv, do, seq_bounds, dqkv)
    L, hd = _packed_dims(qkv, seq_bounds, H)
    for name, t, shape in (("do", do, (L, H * hd)), ("dqkv", dqkv, (L, 3 * H * hd))):
        if t is not None and (t.device != qkv.device or t.dtype != qkv.dtype or tuple(t.shape) != shape):
            raise ValueError("%s must be a %s tensor of shape %s on %s" % (name, qkv.dtype, shape, qkv.device))
    _placed(qkv, device=[("seq_bounds", seq_bounds), ("workspace", workspace)])
    scale = 1.0 / math.sqrt(hd) if scale is None else scale
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv
    nbytes = lib().attn_packed_qkv_workspace_size(_dt(qkv), L, H, hd, 1)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=qkv.device)
    st = lib().attn_packed_qkv_bwd(_dt(qkv), _ptr(qkv), _ptr(do), _ptr(seq_bounds), _ptr(dqkv), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), L, H, hd, float(scale), int(window),
                                   _stream(stream))
    _check(st, "attn_packed_qkv_bwd")
    return dqkv
