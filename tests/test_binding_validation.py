"""The Python binding rejects, before any pointer reaches the library, tensors
the C ABI cannot check itself: host tensors (their addresses would reach the
kernels as device addresses), mixed dtypes, and outputs or side inputs of the
wrong shape, dtype or device.  Runs without a GPU: every case fails first."""
import pytest
import torch

import attention_attn_fwd_08_gb300 as A

B, T, H, Hkv, hd = 2, 8, 4, 2, 64


def t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def qkv():
    return t(B, T, H * hd), t(B, T, Hkv * hd), t(B, T, Hkv * hd)


def test_host_tensors_are_rejected():
    q, k, v = qkv()
    with pytest.raises(ValueError, match="CUDA tensors"):
        A.attn_fwd(q, k, v, H=H, Hkv=Hkv)
    with pytest.raises(ValueError, match="CUDA tensors"):
        A.attn_decode(q[:, -1:].contiguous(), k, v, H=H, Hkv=Hkv)
    with pytest.raises(ValueError, match="CUDA tensors"):
        A.attn_rope(q, H=H)
    cu = torch.tensor([0, 5, 8], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensors"):
        A.attn_varlen_fwd(q[0], k[0], v[0], cu, cu, 5, 5, H=H, Hkv=Hkv)


@pytest.mark.parametrize("case", ["k dtype", "v dtype", "v shape", "o shape", "o dtype", "lse dtype", "lse shape"])
def test_forward_rejects_mismatched_tensors(case):
    q, k, v = qkv()
    kw = dict(H=H, Hkv=Hkv)
    if case == "k dtype":
        k = k.half()
    elif case == "v dtype":
        v = v.float()
    elif case == "v shape":
        v = t(B, T - 1, Hkv * hd)
    elif case == "o shape":
        kw["o"] = t(B, T - 1, H * hd)
    elif case == "o dtype":
        kw["o"] = t(B, T, H * hd, dtype=torch.float16)
    elif case == "lse dtype":
        kw["lse"] = t(B, H, T, dtype=torch.bfloat16)
    else:
        kw["lse"] = t(B, H, T - 1, dtype=torch.float32)
    with pytest.raises(ValueError, match=case.split()[0]):
        A.attn_fwd(q, k, v, **kw)


@pytest.mark.parametrize("name", ["o", "do", "dq", "dk", "dv"])
def test_backward_rejects_mismatched_tensors(name):
    q, k, v = qkv()
    args = dict(o=t(B, T, H * hd), do=t(B, T, H * hd), lse=t(B, H, T, dtype=torch.float32))
    kw = dict(H=H, Hkv=Hkv)
    bad = t(B, T, 1)  # wrong shape for every one of them
    if name in ("o", "do"):
        args[name] = bad
    else:
        kw[name] = bad
    with pytest.raises(ValueError, match=name):
        A.attn_bwd(q, k, v, args["o"], args["do"], args["lse"], **kw)


def test_packed_lse_shape_is_batch_heads_max_rows():
    q, k, v = qkv()
    cu = torch.tensor([0, 5, 8], dtype=torch.int32)
    with pytest.raises(ValueError, match="lse"):
        A.attn_varlen_fwd(q[0], k[0], v[0], cu, cu, 5, 5, H=H, Hkv=Hkv, lse=t(2, H, 8, dtype=torch.float32))
