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
  bf16 (round to nearest even, through fp32) before the attention oracle sees it.
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


def rotate_bf16(x_bf16: torch.Tensor, positions, cos_t, sin_t, rotary_dim: int) -> torch.Tensor:
    """Rotate a bf16 tensor [rows, H, d] in fp64 and round the result to bf16."""
    r = rotate(x_bf16.to(torch.float64).numpy(), positions, np.asarray(cos_t, np.float64),
               np.asarray(sin_t, np.float64), rotary_dim)
    return torch.from_numpy(r).to(torch.float32).to(torch.bfloat16)
