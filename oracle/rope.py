"""RoPE (rotary position embedding) for the oracle — TEST INFRASTRUCTURE ONLY.

The jsqmd page "CANN Transformer算子库ops-transformer深度实践", §三 "RoPE的设计动机与
计算特点", injects position into Q and K by rotating them so that their inner
product depends on the relative position, and decomposes the rotation into
rotations of pairs of adjacent dimensions.  Readings where the pages are silent:

* pairs are (2i, 2i+1) for i < rotary_dim / 2; dimensions >= rotary_dim pass through;
* the angle of pair i at position p comes from caller-given tables,
  cos_t[p, i] and sin_t[p, i] (the page's lookup-table approach, hwcomputing.csdn.net
  page, §1.2); ``tables`` builds the usual ones, angle p * base^(-2i / rotary_dim);
* rotation: (x, y) -> (x cos - y sin, x sin + y cos);
* the rotated Q and K are bf16 tensors (the matmul input precision of the pages,
  hwcomputing.csdn.net page, §2.2), so ``rotate_bf16`` rounds the fp64 result to
  bf16 once, to nearest with ties to even (``bf16_round_bits``), before the
  attention oracle sees it.

Parity status: pinned (tests/test_oracle.py: the tables against the angle
formula, the rotation against a scalar loop, identity at position 0, norm
preservation, relative-position dependence of the scores; the bf16 rounding
against hand-worked ties, neighbours of ties, signed zeros, subnormals and the
overflow threshold, and against a nearest-neighbour search over every finite
bf16 value).
"""

from __future__ import annotations

import numpy as np
import torch


def tables(max_pos: int, rotary_dim: int, base: float = 10000.0):
    """cos/sin tables [max_pos, rotary_dim // 2] in float64."""
    i = np.arange(rotary_dim // 2, dtype=np.float64)
    inv = base ** (-2.0 * i / rotary_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def rotate(x: np.ndarray, positions, cos_t: np.ndarray, sin_t: np.ndarray, rotary_dim: int) -> np.ndarray:
    """x [rows, H, d] float64, positions [rows] -> rotated copy (float64)."""
    out = np.array(x, dtype=np.float64, copy=True)
    pos = np.asarray(positions, dtype=np.int64)
    c = cos_t[pos][:, None, :]          # [rows, 1, rotary_dim/2]
    s = sin_t[pos][:, None, :]
    xe = x[:, :, 0:rotary_dim:2]
    xo = x[:, :, 1:rotary_dim:2]
    out[:, :, 0:rotary_dim:2] = xe * c - xo * s
    out[:, :, 1:rotary_dim:2] = xe * s + xo * c
    return out


def bf16_round_bits(x) -> np.ndarray:
    """Round float64 values to bf16 in one step (nearest, ties to even); return the uint16 bit patterns.

    bf16 is 1 sign bit, 8 exponent bits (bias 127) and 7 stored significand bits.  A normal
    number 2^e' (1 + f) carries 8 significant bits, so the bf16 values next to |x| = m 2^e
    (0.5 <= m < 1) are spaced 2^(e - 8) apart; below the smallest normal, 2^-126, they are the
    subnormals, multiples of 2^-133.  |x| / spacing is rounded to an integer (half to even)
    and scaled back, which is exact in float64; a result of 2^128 or more (|x| at or past the
    midpoint between the largest finite bf16, (2 - 2^-7) 2^127, and 2^128) is infinity.  The
    rounded value is a bf16 number, hence exactly a float32, whose upper 16 bits are the
    pattern.  NaN stays NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(a)                         # a = m 2^e, 0.5 <= m < 1 (e = 0 for a = 0)
        q = np.maximum(e, -125) - 8                # log2 of the bf16 spacing at |x|
        r = np.rint(np.ldexp(a, -q))               # integer multiple of the spacing, ties to even
        y = np.ldexp(r, q)
        y = np.where(y >= 2.0 ** 128, np.inf, y)
        y = np.where(np.isnan(x), np.nan, np.copysign(y, x))
    bits32 = y.astype(np.float32).view(np.uint32)  # exact: every bf16 value is a float32
    return (bits32 >> np.uint32(16)).astype(np.uint16)


def rotate_bf16(x_bf16: torch.Tensor, positions, cos_t, sin_t, rotary_dim: int) -> torch.Tensor:
    """Rotate a bf16 tensor [rows, H, d] in fp64 and round the result to bf16 once (RNE)."""
    r = rotate(x_bf16.to(torch.float64).numpy(), positions, np.asarray(cos_t, np.float64),
               np.asarray(sin_t, np.float64), rotary_dim)
    bits = bf16_round_bits(r)
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
