"""Seeded synthetic workloads shared by the tests, the bench and the oracle runs.

This module only draws inputs and describes shapes; it holds none of the
attention arithmetic.  Every tensor is drawn on the CPU with
``torch.Generator('cpu').manual_seed(seed)`` as float32 ``randn``, optionally
multiplied by a constant, then rounded to bf16.  The same bf16 tensors feed
the CUDA path (after a copy to the device) and the oracle (as bit patterns).

Named workloads (shapes of the models the pages talk about; no weights):

* ``tiny_mha``       B=1, H=2, N=256, d=64, non-causal, scale 1/8
* ``bert_varlen``    B=8, H=12, d=64, per-sequence length uniform in [128, 512]
                     (packed rows + cu_seqlens), non-causal
* ``llama7b_causal`` B=1, Hq=Hkv=32, N=8192, d=128, causal, K drawn x2
* ``gqa_window``     B=4, Hq=32, Hkv=8, N=4096, d=128, causal, window 1024
* ``decode_cache``   B=64, Hq=32, Hkv=8, d=128, cache capacity 8192,
                     per-sequence cache length uniform in [512, 8192]
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch


@dataclass(frozen=True)
class PrefillCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int                      # dense/padded: rows per sequence; packed: max length
    Nk: int
    d: int
    causal: bool = False
    window: int = 0
    seed: int = 0
    layout: str = "dense"        # "dense" | "packed" | "padded"
    len_q: Optional[List[int]] = None   # explicit lengths (packed/padded)
    len_k: Optional[List[int]] = None
    len_range: Optional[tuple] = None   # (lo, hi) inclusive, drawn from the seed
    k_mult: float = 1.0
    scale: Optional[float] = None

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class DecodeCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    Ncap: int
    d: int
    len_range: tuple = (1, 1)            # inclusive, drawn from the seed
    seed: int = 0
    window: int = 0
    lens: Optional[List[int]] = None     # explicit lengths override len_range
    scale: Optional[float] = None

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)


TINY_MHA = PrefillCase("tiny_mha", B=1, Hq=2, Hkv=2, Nq=256, Nk=256, d=64, seed=1, scale=1.0 / 8)
BERT_VARLEN = PrefillCase("bert_varlen", B=8, Hq=12, Hkv=12, Nq=512, Nk=512, d=64, seed=2,
                          layout="packed", len_range=(128, 512))
LLAMA7B_CAUSAL = PrefillCase("llama7b_causal", B=1, Hq=32, Hkv=32, Nq=8192, Nk=8192, d=128,
                             causal=True, seed=3, k_mult=2.0)
GQA_WINDOW = PrefillCase("gqa_window", B=4, Hq=32, Hkv=8, Nq=4096, Nk=4096, d=128,
                         causal=True, window=1024, seed=4)
DECODE_CACHE = DecodeCase("decode_cache", B=64, Hq=32, Hkv=8, Ncap=8192, d=128,
                          len_range=(512, 8192), seed=5)

PREFILL_CASES = {c.name: c for c in (TINY_MHA, BERT_VARLEN, LLAMA7B_CAUSAL, GQA_WINDOW)}


@dataclass
class PrefillInputs:
    case: PrefillCase
    q: torch.Tensor              # bf16, dense/padded [B, Nq, Hq, d]; packed [Tq, Hq, d]
    k: torch.Tensor
    v: torch.Tensor
    len_q: List[int] = field(default_factory=list)
    len_k: List[int] = field(default_factory=list)
    q_off: List[int] = field(default_factory=list)   # first row of each sequence (flattened rows)
    k_off: List[int] = field(default_factory=list)


@dataclass
class DecodeInputs:
    case: DecodeCase
    q: torch.Tensor              # bf16 [B, Hq, d]
    k_cache: torch.Tensor        # bf16 [B, Ncap, Hkv, d]
    v_cache: torch.Tensor
    lens: List[int]


def _randn(g: torch.Generator, shape, mult: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if mult != 1.0:
        x = x * mult
    return x.to(torch.bfloat16)


def make_prefill(case: PrefillCase) -> PrefillInputs:
    g = torch.Generator("cpu").manual_seed(case.seed)
    B = case.B
    if case.layout == "dense":
        len_q, len_k = [case.Nq] * B, [case.Nk] * B
    else:
        if case.len_q is not None:
            len_q = list(case.len_q)
            len_k = list(case.len_k if case.len_k is not None else case.len_q)
        else:
            lo, hi = case.len_range
            lens = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
            len_q, len_k = lens, list(lens)
    if case.layout == "packed":
        tq, tk = sum(len_q), sum(len_k)
        q = _randn(g, (tq, case.Hq, case.d))
        k = _randn(g, (tk, case.Hkv, case.d), case.k_mult)
        v = _randn(g, (tk, case.Hkv, case.d))
        q_off = [0]
        k_off = [0]
        for b in range(B - 1):
            q_off.append(q_off[-1] + len_q[b])
            k_off.append(k_off[-1] + len_k[b])
    else:
        q = _randn(g, (B, case.Nq, case.Hq, case.d))
        k = _randn(g, (B, case.Nk, case.Hkv, case.d), case.k_mult)
        v = _randn(g, (B, case.Nk, case.Hkv, case.d))
        q_off = [b * case.Nq for b in range(B)]
        k_off = [b * case.Nk for b in range(B)]
    return PrefillInputs(case, q, k, v, len_q, len_k, q_off, k_off)


def make_decode(case: DecodeCase) -> DecodeInputs:
    g = torch.Generator("cpu").manual_seed(case.seed)
    if case.lens is not None:
        lens = list(case.lens)
    else:
        lo, hi = case.len_range
        lens = torch.randint(lo, hi + 1, (case.B,), generator=g).tolist()
    q = _randn(g, (case.B, case.Hq, case.d))
    k = _randn(g, (case.B, case.Ncap, case.Hkv, case.d))
    v = _randn(g, (case.B, case.Ncap, case.Hkv, case.d))
    return DecodeInputs(case, q, k, v, lens)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a contiguous bf16 CPU tensor (bit patterns)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def shrink(case, **kw):
    """Same workload family at another size (parity cases)."""
    return replace(case, **kw)
