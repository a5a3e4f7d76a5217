"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle on
the same bf16 inputs, and compare with the acceptance tolerances.

Tolerances (fixed by the acceptance criteria, not tuned): bf16 O max-abs error
<= 1e-2 and relative RMS <= 5e-3; fp32 LSE max-abs error <= 1e-3 where finite;
-inf LSE must match -inf exactly and such rows must be exactly 0.

The named workloads are checked with exactly those numbers (``strict=True``).
Synthetic edge cases with deliberately sharpened scores can produce outputs
|O| > 1.28, where the bf16 output format by itself cannot honour 1e-2: the
round-to-nearest of the stored value alone errs by up to 2^-8 |O| (half an
ulp of an 8-significant-bit format), and rounding the weights P to bf16 adds
at most as much again.  For those cases (``strict=False``) element i may err by
max(1e-2, 2^-7 |O_i|) — identical to 1e-2 wherever |O_i| <= 1.28.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from fa_workloads import DecodeInputs, PrefillInputs, bf16_bits

O_MAX_ABS = 1e-2
O_REL_RMS = 5e-3
LSE_MAX_ABS = 1e-3


def gpu_prefill(x: PrefillInputs, dev="cuda"):
    import flashattention_forward_fa_gb300 as fa
    c = x.case
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    if c.layout == "packed":
        cu_q = torch.tensor([0] + list(np.cumsum(x.len_q)), dtype=torch.int32, device=dev)
        cu_k = torch.tensor([0] + list(np.cumsum(x.len_k)), dtype=torch.int32, device=dev)
        o, lse = fa.fa_fwd_varlen(q, k, v, cu_q, cu_k, max(x.len_q), max(x.len_k), causal=c.causal,
                                  window=c.window, scale=c.softmax_scale,
                                  cu_seqlens_q_host=cu_q.cpu().tolist())
    elif c.layout == "padded":
        sq = torch.tensor(x.len_q, dtype=torch.int32, device=dev)
        sk = torch.tensor(x.len_k, dtype=torch.int32, device=dev)
        o, lse = fa.fa_fwd(q, k, v, causal=c.causal, window=c.window, scale=c.softmax_scale,
                           seqlens_q=sq, seqlens_k=sk)
    else:
        o, lse = fa.fa_fwd(q, k, v, causal=c.causal, window=c.window, scale=c.softmax_scale)
    torch.cuda.synchronize()
    return o, lse


def gather_prefill_rows(x: PrefillInputs, o: torch.Tensor, lse: torch.Tensor, rows: np.ndarray):
    """GPU O/LSE of the given (b, h, i) rows as float64 arrays."""
    oc = o.float().cpu().numpy()
    lc = lse.cpu().numpy()
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    if x.case.layout == "packed":
        r = np.asarray(x.q_off)[b] + i
        return oc[r, h].astype(np.float64), lc[h, r].astype(np.float64)
    return oc[b, i, h].astype(np.float64), lc[b, h, i].astype(np.float64)


def oracle_prefill_rows(x: PrefillInputs, rows: np.ndarray):
    c = x.case
    qf = x.q.reshape(-1, c.Hq, c.d)
    kf = x.k.reshape(-1, c.Hkv, c.d)
    vf = x.v.reshape(-1, c.Hkv, c.d)
    return oracle.attention_rows(bf16_bits(qf), bf16_bits(kf), bf16_bits(vf), x.q_off, x.len_q, x.k_off, x.len_k,
                                 c.softmax_scale, c.causal, c.window, rows)


def sample_rows(x: PrefillInputs, per_head: int, heads=None, seed=0) -> np.ndarray:
    """(b, h, i) rows: tile edges, first/last rows, and random rows of each sequence."""
    rng = np.random.default_rng(seed)
    c = x.case
    heads = range(c.Hq) if heads is None else heads
    out = []
    for b, lq in enumerate(x.len_q):
        if lq == 0:
            continue
        fixed = {0, 1, lq - 1, lq // 2}
        for e in (63, 64, 127, 128, 129, 255, 256, 1023, 1024, 4095, 4096):
            if e < lq:
                fixed.add(e)
        for h in heads:
            rnd = set(rng.integers(0, lq, size=max(0, per_head - len(fixed))).tolist())
            for i in sorted(fixed | rnd):
                out.append((b, h, i))
    return np.asarray(out, dtype=np.int32).reshape(-1, 3)


def check(o_gpu: np.ndarray, l_gpu: np.ndarray, o_ref: np.ndarray, l_ref: np.ndarray, what: str = "",
          strict: bool = True):
    """Assert the acceptance tolerances; return a dict of the measured errors."""
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    empty_ref = np.isneginf(l_ref)
    empty_gpu = np.isneginf(l_gpu)
    assert np.array_equal(empty_ref, empty_gpu), f"{what}: -inf LSE rows differ ({empty_ref.sum()} vs {empty_gpu.sum()})"
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    assert np.all(o_gpu[empty_ref] == 0.0), f"{what}: fully masked rows are not exactly 0"
    fin = ~empty_ref
    res = {"rows": int(len(l_ref)), "empty_rows": int(empty_ref.sum())}
    if fin.any():
        d = o_gpu[fin] - o_ref[fin]
        max_abs = float(np.abs(d).max())
        denom = float(np.sum(o_ref[fin] ** 2))
        rel_rms = math.sqrt(float(np.sum(d ** 2)) / denom) if denom > 0 else 0.0
        lse_err = float(np.abs(l_gpu[fin] - l_ref[fin]).max())
        res.update(o_max_abs=max_abs, o_rel_rms=rel_rms, lse_max_abs=lse_err)
        if strict:
            assert max_abs <= O_MAX_ABS, f"{what}: O max-abs {max_abs:.3e} > {O_MAX_ABS}"
        else:
            bound = np.maximum(O_MAX_ABS, np.abs(o_ref[fin]) * 2.0 ** -7)
            worst = float((np.abs(d) / bound).max())
            res["o_bound_ratio"] = worst
            assert worst <= 1.0, f"{what}: O error exceeds max(1e-2, 2^-7|O|) by x{worst:.3f} (max-abs {max_abs:.3e})"
        assert rel_rms <= O_REL_RMS, f"{what}: O rel-RMS {rel_rms:.3e} > {O_REL_RMS}"
        assert lse_err <= LSE_MAX_ABS, f"{what}: LSE max-abs {lse_err:.3e} > {LSE_MAX_ABS}"
    return res


def gpu_decode(x: DecodeInputs, dev="cuda", num_splits=0, with_host_lens=True, window=None):
    import flashattention_forward_fa_gb300 as fa
    c = x.case
    lens = torch.tensor(x.lens, dtype=torch.int32, device=dev)
    o, lse = fa.fa_decode(x.q.to(dev), x.k_cache.to(dev), x.v_cache.to(dev), lens,
                          window=c.window if window is None else window, scale=c.softmax_scale,
                          num_splits=num_splits, seqlens_k_host=x.lens if with_host_lens else None)
    torch.cuda.synchronize()
    return o, lse


def oracle_decode_rows(x: DecodeInputs, rows: np.ndarray, window=None):
    """rows: (b, h) pairs.  The decode query is row 0 of a 1-row sequence whose keys are
    cache slots 0 .. len-1; with bottom-right causal alignment it sees every one of them."""
    c = x.case
    q4 = x.q.reshape(c.B, 1, c.Hq, c.d)
    trip = np.zeros((len(rows), 3), dtype=np.int32)
    trip[:, 0] = rows[:, 0]
    trip[:, 1] = rows[:, 1]
    return oracle.attention_rows(bf16_bits(q4), bf16_bits(x.k_cache), bf16_bits(x.v_cache),
                                 list(range(c.B)), [1] * c.B, [b * c.Ncap for b in range(c.B)], x.lens,
                                 c.softmax_scale, True, c.window if window is None else window, trip)
