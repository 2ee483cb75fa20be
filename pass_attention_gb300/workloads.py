"""Seeded synthetic inputs and the named workloads.

This module draws random inputs and nothing else: it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from
it without sharing code. Every tensor comes from a ``torch.Generator`` seeded
per workload, on the device the caller names (CPU for the oracle-only tests,
``cuda`` for the GPU path; the oracle then receives a host copy of the same
tensor).

Workloads (sizes and value distributions of the pages' examples and of the
scaled-up measurement cases):

====  ======================================================================
name  inputs
====  ======================================================================
row64         1 x 64 fp32 logits ~ N(0, 1), scale 1.0, blocks of 8 -- the
              curionode page's worked example ("One pass, exactly").
softmax_32k   32768 x 8192 fp32 logits ~ N(0, 1) * 10, row-major, scale 1.0.
attn_4k       B 4, H 16, Sq = Sk = 4096, D 128, bf16 ~ N(0, 1), scale
              1/sqrt(128), non-causal.
attn_causal   B 1, H 32, Sq = Sk = 16384, D 128, bf16 ~ N(0, 1), scale
              1/sqrt(128), causal.
decode_64x32  B 64, H 32, one query, D 128, bf16 ~ N(0, 1), K/V padded to
              Lmax 32768, kv_len[b] ~ U{1..32768}, 16 splits.
====  ======================================================================
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class SoftmaxWorkload:
    name: str
    rows: int
    cols: int
    mult: float      # logits are N(0,1) * mult, drawn in fp32
    scale: float     # softmax scale passed to the kernel
    seed: int


@dataclass(frozen=True)
class AttentionWorkload:
    name: str
    B: int
    H: int
    S: int           # Sq == Sk
    D: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    D: int
    Lmax: int
    num_splits: int
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


ROW64 = SoftmaxWorkload("row64", rows=1, cols=64, mult=1.0, scale=1.0, seed=0)
SOFTMAX_32K = SoftmaxWorkload("softmax_32k", rows=32768, cols=8192, mult=10.0, scale=1.0, seed=1)
ATTN_4K = AttentionWorkload("attn_4k", B=4, H=16, S=4096, D=128, causal=False, seed=2)
ATTN_CAUSAL = AttentionWorkload("attn_causal", B=1, H=32, S=16384, D=128, causal=True, seed=3)
DECODE_64X32 = DecodeWorkload("decode_64x32", B=64, H=32, D=128, Lmax=32768, num_splits=16, seed=4)

WORKLOADS = {w.name: w for w in (ROW64, SOFTMAX_32K, ATTN_4K, ATTN_CAUSAL, DECODE_64X32)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def logits(rows: int, cols: int, mult: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 [rows, cols] drawn i.i.d. N(0, 1) and multiplied by ``mult``."""
    g = _gen(seed, device)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    return x


def qkv(B: int, H: int, Sq: int, Sk: int, D: int, seed: int, device="cpu"):
    """bf16 Q [B,H,Sq,D], K [B,H,Sk,D], V [B,H,Sk,D], i.i.d. N(0, 1) drawn in
    fp32 and rounded to bf16 (round-to-nearest-even)."""
    g = _gen(seed, device)
    out = []
    for S in (Sq, Sk, Sk):
        t = torch.randn((B, H, S, D), generator=g, device=device, dtype=torch.float32)
        out.append(t.to(torch.bfloat16))
    return tuple(out)


def decode_inputs(B: int, H: int, Lmax: int, D: int, seed: int, device="cpu",
                  kv_len=None):
    """Single-query decode inputs.

    Returns q [B,H,D], k [B,H,Lmax,D], v [B,H,Lmax,D] (bf16, i.i.d. N(0,1))
    and kv_len [B] int32 ~ U{1..Lmax} unless ``kv_len`` is given. K and V are
    drawn in slices so that no fp32 copy of the whole cache is ever held.
    """
    g = _gen(seed, device)
    if kv_len is None:
        kv_len = torch.randint(1, Lmax + 1, (B,), generator=g, device=device, dtype=torch.int64)
    kv_len = torch.as_tensor(kv_len, device=device).to(torch.int32)
    q = torch.randn((B, H, D), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    k = torch.empty((B, H, Lmax, D), device=device, dtype=torch.bfloat16)
    v = torch.empty((B, H, Lmax, D), device=device, dtype=torch.bfloat16)
    for t in (k, v):
        for b in range(B):
            t[b] = torch.randn((H, Lmax, D), generator=g, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
    return q, k, v, kv_len
