"""CPU check of the LSE allowance the full-size fused-RoPE test grants for rotated elements at
bf16 rounding boundaries (tests/test_rope_gpu.py, _rope_flip_allowance): on a small causal
problem with a widened margin (so that ~1 % of the rotated elements count as boundary elements),
random patterns of such elements are moved to their other bf16 neighbour in Q and K, the
attention LSE is recomputed in fp64, and every row's change must stay within its allowance.
This pins the Jensen / Hoeffding bound and the choice of the other neighbour."""

import numpy as np
import torch

from fa_workloads import PrefillCase, make_prefill
from oracle import rope as orope
from tests.test_rope_gpu import _near_boundary, _rope_flip_allowance


def _lse_causal(q, k, scale):
    """fp64 LSE of causal rows, q/k [N, H, d] float64 -> [N, H]."""
    n = q.shape[0]
    out = np.zeros((n, q.shape[1]))
    for h in range(q.shape[1]):
        s = scale * q[:, h] @ k[:, h].T
        s[np.triu_indices(n, 1)] = -np.inf
        m = s.max(1)
        out[:, h] = m + np.log(np.exp(s - m[:, None]).sum(1))
    return out


def test_rope_flip_allowance_covers_random_flips():
    case = PrefillCase("flip_check", B=1, Hq=2, Hkv=2, Nq=192, Nk=192, d=64, causal=True, seed=97)
    x = make_prefill(case)
    x.k = (x.k.float() * 2.0).to(torch.bfloat16)          # sharpened, as in llama7b_causal
    rd, H, N, scale = case.d, case.Hq, case.Nq, case.softmax_scale
    pos = np.arange(N)
    tab = np.arange(N, dtype=np.float64)[:, None] * (10000.0 ** (-2.0 * np.arange(rd // 2) / rd))[None, :]
    cos_t = np.cos(tab).astype(np.float32).astype(np.float64)
    sin_t = np.sin(tab).astype(np.float32).astype(np.float64)
    q3, k3 = x.q.reshape(-1, H, case.d), x.k.reshape(-1, H, case.d)
    q_ex = orope.rotate(q3.to(torch.float64).numpy(), pos, cos_t, sin_t, rd)
    k_ex = orope.rotate(k3.to(torch.float64).numpy(), pos, cos_t, sin_t, rd)
    qr = orope.rotate_bf16(q3, pos, cos_t, sin_t, rd)
    kr = orope.rotate_bf16(k3, pos, cos_t, sin_t, rd)
    widen = 2.0 ** 6
    qv, kv = qr.to(torch.float64).numpy(), kr.to(torch.float64).numpy()
    lse0 = _lse_causal(qv, kv, scale)
    allow = _rope_flip_allowance(x, qr, kr, q_ex, k_ex, rd, scale, lse0, widen=widen, max_frac=0.05)
    nq, _ = _near_boundary(q3, q_ex, rd, widen)
    nk, _ = _near_boundary(k3, k_ex, rd, widen)
    assert nq.mean() > 0.002 and nk.mean() > 0.002           # the widened margin flags enough elements
    rng = np.random.default_rng(5)
    q_bits = qr.view(torch.int16).numpy().view(np.uint16)
    k_bits = kr.view(torch.int16).numpy().view(np.uint16)
    worst = 0.0
    for _ in range(12):
        qf, kf = qv.copy(), kv.copy()
        for bits, ex, near, out in ((q_bits, q_ex, nq, qf), (k_bits, k_ex, nk, kf)):
            pick = near & (rng.random(near.shape) < 0.7)
            # the other neighbour: one bf16 step away from the rounding, toward the exact value
            # (bit patterns step by one in magnitude; a larger magnitude is one step up)
            b = bits[..., :rd].astype(np.int32)
            vals = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            up = np.abs(ex[..., :rd]) > np.abs(vals)
            alt = (np.where(up, b + 1, b - 1).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            sub = out[..., :rd]
            sub[pick] = alt[pick]
        d_lse = np.abs(_lse_causal(qf, kf, scale) - lse0)
        worst = max(worst, float((d_lse / allow).max()))
    assert worst <= 1.0, f"an LSE change used {worst:.3f} of its allowance"
    assert worst > 0.01                                       # the flips did move the LSE
