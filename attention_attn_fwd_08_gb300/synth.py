"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws N(0,1) tensors and
key-mask lengths from torch's CPU generator, one fresh generator per tensor
(seed = base + tensor index), and rounds them to the working dtype with
round-to-nearest-even.  Both the CUDA path and the fp64 oracle consume the
same rounded values (the oracle widens them to fp64 exactly).

Workloads (shapes of the attention settings the pages describe):
  fp32_causal     B=1  Tq=Tk=128   H=Hkv=1   hd=64  causal               fp32 forward
  gqa_prefill     B=4  Tq=Tk=2048  H=32 Hkv=8 hd=128 causal               bf16 fwd+bwd
  swa_softcap     B=2  Tq=Tk=8192  H=16 Hkv=4 hd=128 causal window=1024 softcap=50  bf16 fwd+bwd
  encoder_mask    B=8  Tq=Tk=1024  H=Hkv=12  hd=64  bidirectional, per-sequence key mask, fp16 fwd
  decode_lq1/lq4  B=16 Lk=32768 Lq in {1,4} H=32 Hkv=8 hd=128 causal q_offset=Lk-Lq  bf16 decode
  varlen_packed   8 sequences of U{256..2048} rows packed back to back, H=32 Hkv=8 hd=128 causal bf16 fwd+bwd
  gqa_prefill_hd256  B=4 Tq=Tk=2048 H=16 Hkv=4 hd=256 causal  bf16 fwd+bwd
  packed_qkv      16 sequences of U{128..1024} rows packed back to back as fused QKV rows,
                  H=12 hd=64, bidirectional within each sequence, bf16 fwd+bwd
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str
    B: int
    Tq: int
    Tk: int
    H: int
    Hkv: int
    hd: int
    causal: bool
    window: int = 0
    softcap: float = 0.0
    q_offset: int = 0
    key_mask: bool = False  # per-sequence prefix mask with lengths U{Tk/2..Tk}
    backward: bool = False
    decode: bool = False
    seed: int = 0x5EED0000
    notes: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.hd)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "fp32_causal": Workload("fp32_causal", "f32", 1, 128, 128, 1, 1, 64, True, seed=0x5EED0001),
    "gqa_prefill": Workload("gqa_prefill", "bf16", 4, 2048, 2048, 32, 8, 128, True,
                            backward=True, seed=0x5EED0002),
    "swa_softcap": Workload("swa_softcap", "bf16", 2, 8192, 8192, 16, 4, 128, True, window=1024,
                            softcap=50.0, backward=True, seed=0x5EED0003),
    "encoder_mask": Workload("encoder_mask", "f16", 8, 1024, 1024, 12, 12, 64, False,
                             key_mask=True, seed=0x5EED0004),
    "decode_lq1": Workload("decode_lq1", "bf16", 16, 1, 32768, 32, 8, 128, True, q_offset=32767,
                           decode=True, seed=0x5EED0005),
    "decode_lq4": Workload("decode_lq4", "bf16", 16, 4, 32768, 32, 8, 128, True, q_offset=32764,
                           decode=True, seed=0x5EED0006),
    # the GQA prefill's query width (H*hd = 4096) at head size 256
    "gqa_prefill_hd256": Workload("gqa_prefill_hd256", "bf16", 4, 2048, 2048, 16, 4, 256, True,
                                  backward=True, seed=0x5EED0008),
    # Tq/Tk: the bound on a sequence's length (max_seqlen)
    "varlen_packed": Workload("varlen_packed", "bf16", 8, 2048, 2048, 32, 8, 128, True, backward=True,
                              seed=0x5EED0007),
    # encoder batching off a fused QKV projection: B sequences, Tq the longest length
    "packed_qkv": Workload("packed_qkv", "bf16", 16, 1024, 1024, 12, 12, 64, False, backward=True,
                           seed=0x5EED0009),
}


def normal(shape, seed: int, dtype: str = "bf16") -> torch.Tensor:
    """iid N(0,1) from a generator seeded with `seed`, rounded to `dtype` (CPU tensor)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    return x.to(DTYPES[dtype])


def mask_lengths(B: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Per-sequence valid lengths drawn uniformly from the integers [lo, hi]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)


def prefix_mask(lengths: torch.Tensor, Tk: int) -> torch.Tensor:
    """[B, Tk] fp32 key mask, 1 for j < length[b] and 0 after."""
    j = torch.arange(Tk, dtype=torch.int64)
    return (j[None, :] < lengths[:, None]).to(torch.float32)


def make_inputs(w: Workload) -> dict:
    """q, k, v (and dO, key mask) for workload w as CPU tensors in w.dtype."""
    out = {
        "q": normal((w.B, w.Tq, w.H * w.hd), w.seed + 0, w.dtype),
        "k": normal((w.B, w.Tk, w.Hkv * w.hd), w.seed + 1, w.dtype),
        "v": normal((w.B, w.Tk, w.Hkv * w.hd), w.seed + 2, w.dtype),
    }
    if w.backward:
        out["do"] = normal((w.B, w.Tq, w.H * w.hd), w.seed + 3, w.dtype)
    if w.key_mask:
        lens = mask_lengths(w.B, w.Tk // 2, w.Tk, w.seed + 4)
        out["lengths"] = lens
        out["key_mask"] = prefix_mask(lens, w.Tk)
    return out


def make_packed_inputs(w: Workload) -> dict:
    """Packed q, k, v, dO ([total, heads*hd], CPU) for w: w.B sequences with lengths
    drawn uniformly from [256, w.Tq], and their int64 prefix sums ``cu`` (B+1)."""
    lens = mask_lengths(w.B, 256, w.Tq, w.seed + 4)
    cu = torch.zeros(w.B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)
    total = int(cu[-1])
    return {
        "q": normal((total, w.H * w.hd), w.seed + 0, w.dtype),
        "k": normal((total, w.Hkv * w.hd), w.seed + 1, w.dtype),
        "v": normal((total, w.Hkv * w.hd), w.seed + 2, w.dtype),
        "do": normal((total, w.H * w.hd), w.seed + 3, w.dtype),
        "lengths": lens,
        "cu": cu,
    }


def make_packed_qkv_inputs(w: Workload) -> dict:
    """Fused QKV rows [L, 3*H*hd] and dO [L, H*hd] (CPU) for w: w.B sequences with
    lengths drawn uniformly from [w.Tq // 8, w.Tq] packed back to back, each row's
    sequence bounds ``seq_bounds`` (int32 [L, 2]: first row, one past the last row)
    and the lengths."""
    lens = mask_lengths(w.B, w.Tq // 8, w.Tq, w.seed + 4)
    L = int(lens.sum())
    ends = torch.cumsum(lens, 0)
    starts = ends - lens
    seq_bounds = torch.stack([torch.repeat_interleave(starts, lens), torch.repeat_interleave(ends, lens)], 1)
    return {
        "qkv": normal((L, 3 * w.H * w.hd), w.seed + 0, w.dtype),
        "do": normal((L, w.H * w.hd), w.seed + 3, w.dtype),
        "seq_bounds": seq_bounds.to(torch.int32).contiguous(),
        "lengths": lens,
    }
