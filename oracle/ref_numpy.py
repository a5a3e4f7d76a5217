"""Independent fp64 numpy oracle — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  It shares no code with the CUDA path and none
with ``attention_ref.c`` (the two oracles cross-check each other).

``attention`` materialises the whole score matrix of one (sequence, head) the
way the naive formulation does — the jsqmd page "CANN Transformer算子库
ops-transformer深度实践", §二 "SelfAttention的基础实现与瓶颈" and its
``naive_attention`` sketch; the agent.csdn.net BERT walkthrough, 第一章
(``BertSelfAttention.forward``: scores = QK^T/sqrt(d) + mask, softmax, times V).
The softmax subtracts the row max first, as the hwcomputing.csdn.net page,
§2.2 "数值稳定性优化", prescribes.

``merge_partials`` is the log-sum-exp merge of attention computed over
disjoint key subsets (split-KV decode combine).  The pages do not print it;
it is the identity that lets the running-max/running-sum softmax of the
hwcomputing.csdn.net page, §2.2 (local block maxima corrected by a global max),
be evaluated in pieces: with lse_s = log sum_{j in s} exp(s_j),
LSE = log sum_s exp(lse_s) and O = sum_s exp(lse_s - LSE) O_s.

Readings (causal alignment, window, GQA head map, empty rows, LSE units) are
the same as in ``attention_ref.c``; they are spelled out there and in the
design notes.
"""

from __future__ import annotations

import numpy as np


def visible_mask(lq: int, lk: int, causal: bool, window: int) -> np.ndarray:
    """Boolean [lq, lk] matrix: may query row i see key j?

    Row i sits at absolute position p = i + lk - lq (bottom-right alignment).
    """
    p = np.arange(lq)[:, None] + (lk - lq)
    j = np.arange(lk)[None, :]
    vis = np.ones((lq, lk), dtype=bool)
    if causal:
        vis &= j <= p
        if window > 0:
            vis &= j > p - window
    elif window > 0:
        vis &= np.abs(p - j) < window
    return vis


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
              causal: bool = False, window: int = 0, alibi_slopes=None):
    """One sequence.  q [lq, Hq, d], k/v [lk, Hkv, d] (float64).

    alibi_slopes: optional [Hq] slopes; the jsqmd page's ALiBi (§三) adds -m_h |p - j|
    to each scaled score, p the query's absolute position (bottom-right aligned).
    Returns O [lq, Hq, d] and LSE [Hq, lq] (float64).
    """
    lq, hq, d = q.shape
    lk, hkv, _ = k.shape
    assert hq % hkv == 0
    group = hq // hkv
    vis = visible_mask(lq, lk, causal, window)
    dist = np.abs((np.arange(lq)[:, None] + (lk - lq)) - np.arange(lk)[None, :]).astype(np.float64)
    o = np.zeros((lq, hq, d))
    lse = np.full((hq, lq), -np.inf)
    for h in range(hq):
        g = h // group
        s = (q[:, h, :] @ k[:, g, :].T) * scale          # [lq, lk]
        if alibi_slopes is not None:
            s = s - alibi_slopes[h] * dist
        s = np.where(vis, s, -np.inf)
        has_key = vis.any(axis=1)
        m = np.where(has_key, s.max(axis=1, initial=-np.inf), 0.0)
        e = np.where(vis, np.exp(s - m[:, None]), 0.0)
        z = e.sum(axis=1)
        p = np.divide(e, z[:, None], out=np.zeros_like(e), where=has_key[:, None])
        o[:, h, :] = p @ v[:, g, :]
        lse[h] = np.where(has_key, m + np.log(np.where(has_key, z, 1.0)), -np.inf)
    return o, lse


def merge_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge S partial results over disjoint key subsets.

    o_parts [S, ..., d] (each normalised over its own subset), lse_parts [S, ...].
    Subsets with lse = -inf (no key) contribute nothing.  Returns (O, LSE).
    """
    mx = lse_parts.max(axis=0)
    finite = np.isfinite(mx)
    base = np.where(finite, mx, 0.0)
    w = np.exp(lse_parts - base[None])                   # exp(-inf) = 0
    tot = w.sum(axis=0)
    lse = np.where(finite, base + np.log(np.where(finite, tot, 1.0)), -np.inf)
    wn = np.divide(w, tot[None], out=np.zeros_like(w), where=finite[None])
    o = (wn[..., None] * o_parts).sum(axis=0)
    return o, lse
