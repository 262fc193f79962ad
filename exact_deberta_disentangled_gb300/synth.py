"""Seeded synthetic inputs for the disentangled-attention workloads.

This module holds no arithmetic of the attention method: it only draws
random tensors, padding lengths and packed-sequence offsets, so that the CUDA
path, the oracle-based tests and the benchmark all see the same inputs.

Recipe (one ``torch.Generator`` per workload, seeded with the workload's
index): fp32 ``randn`` in the order Q, K, V, Qr, Kr, dO, then cast to the
compute dtype; padding lengths or packed sequence lengths are drawn from the
same generator afterwards.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@dataclass
class Workload:
    name: str
    H: int
    D: int
    span: int
    nb: int
    mp: int
    dtype: str
    seed: int
    B: int = 0                 # padded: number of sequences
    L: int = 0                 # padded: sequence length (packed: max length)
    total_tokens: int = 0      # packed only
    packed: bool = False
    len_range: Optional[tuple] = None   # padded: valid-length range; packed: sequence-length range
    dropout_p: float = 0.0

    @property
    def R(self) -> int:
        return 2 * self.span


def _workloads():
    w = {}
    w["tiny_fp32"] = Workload("tiny_fp32", H=2, D=64, span=64, nb=64, mp=128, dtype="fp32", seed=0, B=1, L=128)
    w["v3_base"] = Workload("v3_base", H=12, D=64, span=256, nb=256, mp=512, dtype="bf16", seed=1, B=32, L=512,
                            len_range=(256, 512))
    for L in (512, 1024, 2048, 4096, 8192):
        w[f"sweep_L{L}"] = Workload(f"sweep_L{L}", H=12, D=64, span=256, nb=256, mp=512, dtype="bf16", seed=2,
                                    B=16384 // L, L=L)
    w["varlen"] = Workload("varlen", H=12, D=64, span=256, nb=256, mp=512, dtype="bf16", seed=3, packed=True,
                           total_tokens=16384, len_range=(32, 2048))
    w["hd128_dropout"] = Workload("hd128_dropout", H=8, D=128, span=256, nb=256, mp=512, dtype="bf16", seed=4,
                                  B=4, L=4096, dropout_p=0.1)
    w["hd32_dropout"] = Workload("hd32_dropout", H=24, D=32, span=256, nb=256, mp=512, dtype="bf16", seed=4,
                                 B=8, L=2048, dropout_p=0.1)
    # stand-in for the pages' MNLI evaluation shape (fp16, batch 8, length
    # bucket 512, a 24-head / 64-dim model): padded batches of 8 sequences
    # with valid lengths uniform in [16, 512]; synthetic values, no dataset
    w["mnli_fp16"] = Workload("mnli_fp16", H=24, D=64, span=256, nb=256, mp=512, dtype="fp16", seed=5, B=8,
                              L=512, len_range=(16, 512))
    return w


WORKLOADS = _workloads()


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    qr: torch.Tensor
    kr: torch.Tensor
    dout: torch.Tensor
    cu_seqlens: torch.Tensor          # int32 [nseq + 1]
    qmask: Optional[torch.Tensor]     # uint8 [T] (padded layout only) or None
    kmask: Optional[torch.Tensor]
    B: int                            # number of sequences
    L: int                            # padded length, or the longest packed sequence
    packed: bool
    extra: dict = field(default_factory=dict)


def packed_lengths(gen: torch.Generator, total: int, lo: int, hi: int) -> list:
    """Sequence lengths drawn uniformly in [lo, hi] until they cover ``total``
    tokens; the last one is cut to the remainder."""
    out, acc = [], 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def make_inputs(w: Workload, *, B: Optional[int] = None, L: Optional[int] = None, H: Optional[int] = None,
                total_tokens: Optional[int] = None, dtype: Optional[str] = None, seed: Optional[int] = None,
                key_mask: str = "same", device="cpu") -> Inputs:
    """Draw the inputs of workload ``w`` (optionally at reduced sizes for the
    small parity cases; the recipe stays the same).

    ``key_mask`` (padded workloads with a length range only): "same" makes the
    key mask equal to the query mask (the workloads' recipe); "independent"
    draws, after everything else, a second set of valid lengths for the keys
    and then clears about one key in eight at random inside them, so that the
    two masks differ both at the padding boundary and in scattered positions."""
    B = w.B if B is None else B
    L = w.L if L is None else L
    H = w.H if H is None else H
    dt = DTYPES[w.dtype if dtype is None else dtype]
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    if w.packed:
        T = w.total_tokens if total_tokens is None else total_tokens
    else:
        T = B * L
    shape = (T, H, w.D)
    q = torch.randn(shape, generator=gen)
    k = torch.randn(shape, generator=gen)
    v = torch.randn(shape, generator=gen)
    qr = torch.randn((H, w.R, w.D), generator=gen)
    kr = torch.randn((H, w.R, w.D), generator=gen)
    dout = torch.randn(shape, generator=gen)
    qmask = kmask = None
    if w.packed:
        lo, hi = w.len_range
        lens = packed_lengths(gen, T, lo, hi)
        cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int32), 0)
        nseq, Lmax = len(lens), max(lens)
    else:
        cu = torch.arange(0, B + 1, dtype=torch.int32) * L
        nseq, Lmax = B, L
        if w.len_range is not None:
            lo, hi = w.len_range
            lo, hi = min(lo, L), min(hi, L)
            lens = torch.randint(lo, hi + 1, (B,), generator=gen)
            pos = torch.arange(L)[None, :]
            m = (pos < lens[:, None]).to(torch.uint8).reshape(-1)
            qmask = m.clone()
            kmask = m.clone()
            if key_mask == "independent":
                klens = torch.randint(lo, hi + 1, (B,), generator=gen)
                km = (pos < klens[:, None]).reshape(-1)
                holes = torch.rand(B * L, generator=gen) < 0.125
                kmask = (km & ~holes).to(torch.uint8)
            elif key_mask != "same":
                raise ValueError(f"key_mask must be 'same' or 'independent', not {key_mask!r}")
    t = [x.to(dt).to(device) for x in (q, k, v, qr, kr, dout)]
    cu = cu.to(device)
    if qmask is not None:
        qmask, kmask = qmask.to(device), kmask.to(device)
    return Inputs(*t, cu_seqlens=cu, qmask=qmask, kmask=kmask, B=nseq, L=Lmax, packed=w.packed)
