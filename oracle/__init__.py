"""fp64 CPU attention oracle -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline /
reference arm may import this package.  The product library never does, and
this package imports nothing from it: the two share no code.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, one materialised
probability row per query); this module compiles it with gcc and marshals
numpy arrays through ctypes.  Every function here follows the definition
written at the top of ``attn_oracle.c``, which cites the pages it restates:

* ferrotensor_backend engine/attention.rs -- AttentionOptions (causal offset,
  window predicate), AttentionDims (head_dim, GQA divisibility, 1/sqrt(hd)).
* brotensor ops/flash_attention.h -- key mask (> 0.5 keeps a key), softcap
  position, GQA head map, decode row positions, overwrite semantics.
* vision_rs flash_attn2.rs -- forward with saved log-sum-exp, dQ and dK/dV.
* forge attention.metal -- unfused forward with materialised P, D = dO.O,
  softcap derivative, GQA group sums in dK/dV.

Pins: every function here is checked against closed forms, invariants, an
independent torch fp64 route and finite differences in
``tests/test_oracle_pins.py``.  One reading is a choice among conflicting
pages rather than a fixed fact: the non-causal sliding window (ferrotensor's
``|p - j| < window``); its implementation is pinned to that formula, the choice
of formula is recorded as a reading.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into a shared library (gcc, OpenMP). Returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        common = [ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                       ctypes.c_longlong, dp, ctypes.c_longlong]
        lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp] + common
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_probs.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_int] + common
        lib.oracle_attn_probs.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [dp] * 7 + common
        lib.oracle_attn_bwd.restype = ctypes.c_int
        llp = ctypes.POINTER(ctypes.c_longlong)
        common_ex = [ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_double,
                                          ctypes.c_longlong, dp, ctypes.c_longlong, dp, llp]
        lib.oracle_attn_fwd_ex.argtypes = [dp, dp, dp, dp, dp] + common_ex
        lib.oracle_attn_fwd_ex.restype = ctypes.c_int
        lib.oracle_attn_probs_ex.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_int] + common_ex
        lib.oracle_attn_probs_ex.restype = ctypes.c_int
        lib.oracle_attn_bwd_ex.argtypes = [dp] * 7 + common_ex
        lib.oracle_attn_bwd_ex.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shapes(q, k, H, Hkv):
    if q.ndim != 3 or k.ndim != 3:
        raise ValueError("q must be [B,Tq,H*hd] and k/v [B,Tk,Hkv*hd]")
    B, Tq, qc = q.shape
    _, Tk, kc = k.shape
    if qc % H or kc % Hkv or qc // H != kc // Hkv:
        raise ValueError("inconsistent head sizes")
    return B, Tq, Tk, qc // H


def _mask(key_mask, B, Tk):
    """Returns (array or None, batch stride). A 1-D mask is shared by every batch."""
    if key_mask is None:
        return None, 0
    m = _f64(key_mask)
    if m.ndim == 1:
        if m.shape[0] != Tk:
            raise ValueError("key mask must have Tk entries")
        return m, 0
    if m.shape != (B, Tk):
        raise ValueError("key mask must be [Tk] or [B,Tk]")
    return m, Tk


def _common(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, m, ms):
    return [B, Tq, Tk, H, Hkv, hd, float(scale), int(bool(causal)), int(window), float(softcap),
            int(q_offset), _ptr(m), int(ms)]


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().oracle_num_threads())


def fwd(q, k, v, *, H, Hkv, scale, causal=False, window=0, softcap=0.0, q_offset=0,
        key_mask=None):
    """O [B,Tq,H*hd] and LSE [B,H,Tq] of the plain definition (fp64)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Tq, Tk, hd = _shapes(q, k, H, Hkv)
    m, ms = _mask(key_mask, B, Tk)
    o = np.zeros((B, Tq, H * hd), np.float64)
    lse = np.zeros((B, H, Tq), np.float64)
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 *_common(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap,
                                          q_offset, m, ms))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse


def probs(q, k, v, b, h, *, H, Hkv, scale, causal=False, window=0, softcap=0.0, q_offset=0,
          key_mask=None):
    """The materialised probability matrix P [Tq,Tk] of batch b, head h."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Tq, Tk, hd = _shapes(q, k, H, Hkv)
    m, ms = _mask(key_mask, B, Tk)
    P = np.zeros((Tq, Tk), np.float64)
    rc = _load().oracle_attn_probs(_ptr(q), _ptr(k), _ptr(v), _ptr(P), int(b), int(h),
                                   *_common(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap,
                                            q_offset, m, ms))
    if rc != 0:
        raise ValueError("oracle_attn_probs rejected its arguments")
    return P


def bwd(q, k, v, do, *, H, Hkv, scale, causal=False, window=0, softcap=0.0, q_offset=0,
        key_mask=None):
    """dQ, dK, dV of the plain definition, with P rebuilt from the inputs."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Tq, Tk, hd = _shapes(q, k, H, Hkv)
    if do.shape != q.shape:
        raise ValueError("dO must have q's shape")
    m, ms = _mask(key_mask, B, Tk)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                                 *_common(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap,
                                          q_offset, m, ms))
    if rc != 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return dq, dk, dv


def _bias(bias, B, H, Tq, Tk):
    """(array or None, 4 strides): an additive bias broadcastable to [B, H, Tq, Tk],
    size-1 dimensions read with stride 0 (ferrotensor engine/attention.rs, mask_strides)."""
    if bias is None:
        return None, None
    a = _f64(bias)
    if a.ndim != 4:
        raise ValueError("bias must be 4-D [B|1, H|1, Tq|1, Tk|1]")
    full = (B, H, Tq, Tk)
    st = []
    for dim, n, sb in zip(a.shape, full, a.strides):
        if dim not in (1, n):
            raise ValueError("bias shape %s does not broadcast to %s" % (a.shape, full))
        st.append(0 if dim == 1 else sb // 8)
    return a, (ctypes.c_longlong * 4)(*st)


def _common_ex(B, Tq, Tk, H, Hkv, hd, scale, wl, wr, softcap, q_offset, m, ms, bias, bs):
    return [B, Tq, Tk, H, Hkv, hd, float(scale), int(wl), int(wr), float(softcap), int(q_offset), _ptr(m), int(ms),
            _ptr(bias), bs]


def fwd_ex(q, k, v, *, H, Hkv, scale, window_left=-1, window_right=-1, softcap=0.0, q_offset=0, key_mask=None,
           bias=None):
    """O and LSE with the two-sided window [p - window_left, p + window_right]
    (negative = unbounded) and an optional additive bias (see attn_oracle.c)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Tq, Tk, hd = _shapes(q, k, H, Hkv)
    m, ms = _mask(key_mask, B, Tk)
    bb, bs = _bias(bias, B, H, Tq, Tk)
    o = np.zeros((B, Tq, H * hd), np.float64)
    lse = np.zeros((B, H, Tq), np.float64)
    rc = _load().oracle_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                    *_common_ex(B, Tq, Tk, H, Hkv, hd, scale, window_left, window_right, softcap,
                                                q_offset, m, ms, bb, bs))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_ex rejected its arguments")
    return o, lse


def probs_ex(q, k, v, b, h, *, H, Hkv, scale, window_left=-1, window_right=-1, softcap=0.0, q_offset=0,
             key_mask=None, bias=None):
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Tq, Tk, hd = _shapes(q, k, H, Hkv)
    m, ms = _mask(key_mask, B, Tk)
    bb, bs = _bias(bias, B, H, Tq, Tk)
    P = np.zeros((Tq, Tk), np.float64)
    rc = _load().oracle_attn_probs_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(P), int(b), int(h),
                                      *_common_ex(B, Tq, Tk, H, Hkv, hd, scale, window_left, window_right, softcap,
                                                  q_offset, m, ms, bb, bs))
    if rc != 0:
        raise ValueError("oracle_attn_probs_ex rejected its arguments")
    return P


def bwd_ex(q, k, v, do, *, H, Hkv, scale, window_left=-1, window_right=-1, softcap=0.0, q_offset=0, key_mask=None,
           bias=None):
    """dQ, dK, dV of fwd_ex (the bias is a constant: it enters through P only)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Tq, Tk, hd = _shapes(q, k, H, Hkv)
    m, ms = _mask(key_mask, B, Tk)
    bb, bs = _bias(bias, B, H, Tq, Tk)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    rc = _load().oracle_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                                    *_common_ex(B, Tq, Tk, H, Hkv, hd, scale, window_left, window_right, softcap,
                                                q_offset, m, ms, bb, bs))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_ex rejected its arguments")
    return dq, dk, dv


def varlen_fwd(q, k, v, cu_q, cu_k, *, H, Hkv, scale, causal=False, window=0, softcap=0.0):
    """Packed variable-length forward (brotensor ops/flash_attention.h,
    flash_attention_varlen_forward): sequence b is rows cu_q[b] .. cu_q[b+1]-1 of
    q [total_q, H*hd] and rows cu_k[b] .. cu_k[b+1]-1 of k/v, attended to as its
    own batch of one with query positions counted from its first row; nothing
    crosses sequences.  Returns O [total_q, H*hd] (zero on rows outside every
    sequence) and LSE as a list of [H, Tq_b] arrays, one per sequence."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    hd = q.shape[1] // H
    o = np.zeros_like(q)
    lses = []
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if q1 == q0:
            lses.append(np.zeros((H, 0)))
            continue
        if k1 == k0:  # no key at all: every row fully masked (O = 0, LSE = -inf)
            lses.append(np.full((H, q1 - q0), -np.inf))
            continue
        ob, lb = fwd(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], H=H, Hkv=Hkv, scale=scale, causal=causal,
                     window=window, softcap=softcap)
        o[q0:q1] = ob[0]
        lses.append(lb[0])
    return o, lses


def varlen_bwd(q, k, v, do, cu_q, cu_k, *, H, Hkv, scale, causal=False, window=0, softcap=0.0):
    """Backward of varlen_fwd (brotensor flash_attention_varlen_backward: the
    per-sequence backward; excluded positions contribute nothing).  Returns dQ,
    dK, dV on the packed rows, zero outside every sequence."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if q1 == q0 or k1 == k0:
            continue
        gq, gk, gv = bwd(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], do[None, q0:q1], H=H, Hkv=Hkv, scale=scale,
                         causal=causal, window=window, softcap=softcap)
        dq[q0:q1], dk[k0:k1], dv[k0:k1] = gq[0], gk[0], gv[0]
    return dq, dk, dv


def rope(x, *, head_dim, pos=0, theta=10000.0):
    """Rotate-half rotary embedding (ferrotensor engine/attention.rs, rope /
    rope_theta): x is [batch, seq, heads*head_dim]; every head vector of token s
    (counted within its sequence) gets position pos + s, and its pair
    (x[i], x[i + head_dim/2]), i < head_dim/2, turns by the angle
    (pos + s) * theta**(-2i/head_dim):
        x'[i]          = x[i] cos - x[i + head_dim/2] sin
        x'[i + hd/2]   = x[i + head_dim/2] cos + x[i] sin
    Returns a new fp64 array (the page rotates in place)."""
    x = _f64(x)
    B, T, C = x.shape
    hd = int(head_dim)
    if hd % 2 or C % hd:
        raise ValueError("head_dim must be even and divide the row")
    half = hd // 2
    out = x.copy().reshape(B, T, C // hd, hd)
    xin = x.reshape(B, T, C // hd, hd)
    for s in range(T):
        p = float(pos + s)
        for i in range(half):
            ang = p * float(theta) ** (-2.0 * i / hd)
            c, sn = np.cos(ang), np.sin(ang)
            a, b = xin[:, s, :, i], xin[:, s, :, i + half]
            out[:, s, :, i] = a * c - b * sn
            out[:, s, :, i + half] = b * c + a * sn
    return out.reshape(B, T, C)


def _packed_rows(seq_bounds, L, window):
    """Visible keys of every row of a packed fused-QKV batch: row r attends keys j of
    its own sequence, seq_bounds[r, 0] <= j < seq_bounds[r, 1], and with window > 0
    only those with |r - j| <= window // 2 (brotensor ops/flash_attention.h,
    flash_attention_packed_qkv_forward)."""
    sb = np.asarray(seq_bounds, dtype=np.int64).reshape(L, 2)
    rows = []
    for r in range(L):
        j = np.arange(max(int(sb[r, 0]), 0), min(int(sb[r, 1]), L))
        if window > 0:
            j = j[np.abs(r - j) <= window // 2]
        rows.append(j)
    return rows


def _split_qkv(qkv, H):
    qkv = _f64(qkv)
    L, C = qkv.shape
    hd = C // (3 * H)
    if 3 * H * hd != C:
        raise ValueError("qkv rows must hold 3 * H * head_dim values")
    return (qkv[:, :H * hd].reshape(L, H, hd), qkv[:, H * hd:2 * H * hd].reshape(L, H, hd),
            qkv[:, 2 * H * hd:].reshape(L, H, hd), L, hd)


def packed_qkv_fwd(qkv, seq_bounds, *, H, scale, window=0):
    """Packed bidirectional self-attention straight off a fused QKV projection
    (brotensor ops/flash_attention.h, flash_attention_packed_qkv_forward): qkv is
    [L, 3*H*hd], each row [q heads | k heads | v heads]; the visible keys of row r
    are those of _packed_rows.  Written out row by row in numpy fp64 (independent of
    attn_oracle.c).  Returns O [L, H*hd] and LSE [H, L] (-inf for a row that sees
    no key, whose O is 0)."""
    q, k, v, L, hd = _split_qkv(qkv, H)
    o = np.zeros((L, H, hd))
    lse = np.full((H, L), -np.inf)
    for r, j in enumerate(_packed_rows(seq_bounds, L, window)):
        if j.size == 0:
            continue
        s = scale * np.einsum("hd,jhd->hj", q[r], k[j])  # [H, keys]
        mx = s.max(axis=1, keepdims=True)
        p = np.exp(s - mx)
        l = p.sum(axis=1, keepdims=True)
        o[r] = np.einsum("hj,jhd->hd", p / l, v[j])
        lse[:, r] = (mx + np.log(l))[:, 0]
    return o.reshape(L, H * hd), lse


def packed_qkv_bwd(qkv, do, seq_bounds, *, H, scale, window=0):
    """Backward of packed_qkv_fwd (brotensor flash_attention_packed_qkv_backward):
    dQKV [L, 3*H*hd], each row [dQ heads | dK heads | dV heads].  Per row r and head:
    P = softmax(scale * q_r . k_j) over its visible keys, dP_j = dO_r . v_j,
    dS = P (dP - sum(P dP)), dq_r = scale * sum_j dS_j k_j, dk_j += scale * dS_j q_r,
    dv_j += P_j dO_r; row by row in numpy fp64."""
    q, k, v, L, hd = _split_qkv(qkv, H)
    do = _f64(do).reshape(L, H, hd)
    dq, dk, dv = np.zeros((L, H, hd)), np.zeros((L, H, hd)), np.zeros((L, H, hd))
    for r, j in enumerate(_packed_rows(seq_bounds, L, window)):
        if j.size == 0:
            continue
        s = scale * np.einsum("hd,jhd->hj", q[r], k[j])
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        dp = np.einsum("hd,jhd->hj", do[r], v[j])
        ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        dq[r] = scale * np.einsum("hj,jhd->hd", ds, k[j])
        dk[j] += scale * np.einsum("hj,hd->jhd", ds, q[r])
        dv[j] += np.einsum("hj,hd->jhd", p, do[r])
    return np.concatenate([dq.reshape(L, -1), dk.reshape(L, -1), dv.reshape(L, -1)], axis=1)
