"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle on
the same bf16 inputs, and compare with the acceptance tolerances.

The rule (one for every test):

* Strict (``strict=True``), the acceptance numbers as written: bf16 O max-abs
  error <= 1e-2 and relative RMS <= 5e-3; fp32 LSE max-abs error <= 1e-3 where
  finite; -inf LSE must match -inf exactly and such rows must be exactly 0.
  Every named workload (tiny_mha, bert_varlen, llama7b_causal, gqa_window,
  decode_cache, at full size and every row) and every fixed-shape case with
  unsharpened N(0, 1) inputs is held to it.

* Derived (``strict=False``), for inputs that can push outputs to |O| > 1.28
  (few visible keys, sharpened or rising scores, random draws of those): the
  same RMS, LSE and masked-row rules, but element i of O may err by
      max(1e-2, 1.125 * 2^-8 * (|O_i| + A_i)),   A_i = sum_j p_ij |v_jt|,
  i.e. 1e-2, or, where the bf16 format cannot honour 1e-2, what the kernel's
  two bf16 roundings imply: the weights p_ij enter P V rounded to bf16
  (relative error <= 2^-8 each, which moves O_i by at most 2^-8 A_i), and O is
  stored as bf16 (at most 2^-8 |O_i|); the factor 1.125 covers the fp32 sums,
  ex2.approx and the division.  A_i is the oracle's attention over |V| (the
  same weights applied to the absolute values), computed alongside.  The
  returned measures count how many elements needed the derived side
  (``o_loose_elems``: error above 1e-2).
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
DERIVED_FACTOR = 1.125 * 2.0 ** -8


def abs_bits(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of |x| (clear the sign bit; exact)."""
    return np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)


def gpu_prefill(x: PrefillInputs, dev="cuda", out=None, lse=None):
    import flashattention_forward_fa_gb300 as fa
    c = x.case
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    if c.layout == "packed":
        cu_q = torch.tensor([0] + list(np.cumsum(x.len_q)), dtype=torch.int32, device=dev)
        cu_k = torch.tensor([0] + list(np.cumsum(x.len_k)), dtype=torch.int32, device=dev)
        o, lse = fa.fa_fwd_varlen(q, k, v, cu_q, cu_k, max(x.len_q), max(x.len_k), causal=c.causal,
                                  window=c.window, scale=c.softmax_scale,
                                  cu_seqlens_q_host=cu_q.cpu().tolist(), out=out, lse=lse)
    elif c.layout == "padded":
        sq = torch.tensor(x.len_q, dtype=torch.int32, device=dev)
        sk = torch.tensor(x.len_k, dtype=torch.int32, device=dev)
        o, lse = fa.fa_fwd(q, k, v, causal=c.causal, window=c.window, scale=c.softmax_scale,
                           seqlens_q=sq, seqlens_k=sk, out=out, lse=lse)
    else:
        o, lse = fa.fa_fwd(q, k, v, causal=c.causal, window=c.window, scale=c.softmax_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    return o, lse


def host_outputs(o: torch.Tensor, lse: torch.Tensor):
    """O and LSE as host float32 arrays (converted once; rows are then gathered by index)."""
    return o.float().cpu().numpy(), lse.cpu().numpy()


def gather_prefill_rows(x: PrefillInputs, o, lse, rows: np.ndarray):
    """GPU O/LSE of the given (b, h, i) rows as float64 arrays (o, lse: tensors or host arrays)."""
    oc = o.float().cpu().numpy() if isinstance(o, torch.Tensor) else o
    lc = lse.cpu().numpy() if isinstance(lse, torch.Tensor) else lse
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    if x.case.layout == "packed":
        r = np.asarray(x.q_off)[b] + i
        return oc[r, h].astype(np.float64), lc[h, r].astype(np.float64)
    return oc[b, i, h].astype(np.float64), lc[b, h, i].astype(np.float64)


class PrefillOracle:
    """The oracle over one set of prefill inputs, with the bf16 bit patterns converted once."""

    def __init__(self, x: PrefillInputs, alibi_slopes=None):
        c = x.case
        self.x = x
        self.q = bf16_bits(x.q.reshape(-1, c.Hq, c.d))
        self.k = bf16_bits(x.k.reshape(-1, c.Hkv, c.d))
        self.v = bf16_bits(x.v.reshape(-1, c.Hkv, c.d))
        self.slopes = None if alibi_slopes is None else np.asarray(alibi_slopes, np.float64)

    def rows(self, rows: np.ndarray, abs_v: bool = False):
        x, c = self.x, self.x.case
        return oracle.attention_rows(self.q, self.k, abs_bits(self.v) if abs_v else self.v, x.q_off, x.len_q,
                                     x.k_off, x.len_k, c.softmax_scale, c.causal, c.window, rows,
                                     alibi_slopes=self.slopes)


def oracle_prefill_rows(x: PrefillInputs, rows: np.ndarray, abs_v: bool = False, alibi_slopes=None):
    return PrefillOracle(x, alibi_slopes).rows(rows, abs_v)


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


class Parity:
    """The acceptance measures, accumulated over chunks of rows (so a full-size workload can be
    compared row by row without holding every oracle row at once).  ``add`` checks the per-row
    rules as it goes; ``result`` checks the aggregate ones and returns the measures."""

    def __init__(self, what: str = "", strict: bool = True):
        self.what, self.strict = what, strict
        self.rows = self.empty = self.loose = 0
        self.max_abs = self.lse_err = self.ratio = 0.0
        self.sq_err = self.sq_ref = 0.0

    def add(self, o_gpu, l_gpu, o_ref, l_ref, o_abs=None):
        what = self.what
        assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
        empty_ref = np.isneginf(l_ref)
        empty_gpu = np.isneginf(l_gpu)
        assert np.array_equal(empty_ref, empty_gpu), \
            f"{what}: -inf LSE rows differ ({empty_ref.sum()} vs {empty_gpu.sum()})"
        assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
        assert np.all(o_gpu[empty_ref] == 0.0), f"{what}: fully masked rows are not exactly 0"
        self.rows += int(len(l_ref))
        self.empty += int(empty_ref.sum())
        fin = ~empty_ref
        if not fin.any():
            return
        d = np.abs(o_gpu[fin] - o_ref[fin])
        self.max_abs = max(self.max_abs, float(d.max()))
        self.sq_err += float(np.sum(d ** 2))
        self.sq_ref += float(np.sum(o_ref[fin] ** 2))
        self.lse_err = max(self.lse_err, float(np.abs(l_gpu[fin] - l_ref[fin]).max()))
        self.loose += int((d > O_MAX_ABS).sum())
        if not self.strict:
            assert o_abs is not None, f"{what}: the derived bound needs the oracle's attention over |V|"
            bound = np.maximum(O_MAX_ABS, DERIVED_FACTOR * (np.abs(o_ref[fin]) + o_abs[fin]))
            self.ratio = max(self.ratio, float((d / bound).max()))

    def result(self) -> dict:
        what = self.what
        res = {"rows": self.rows, "empty_rows": self.empty}
        if self.rows == self.empty:
            return res
        rel_rms = math.sqrt(self.sq_err / self.sq_ref) if self.sq_ref > 0 else 0.0
        res.update(o_max_abs=self.max_abs, o_rel_rms=rel_rms, lse_max_abs=self.lse_err, o_loose_elems=self.loose)
        if self.strict:
            assert self.max_abs <= O_MAX_ABS, f"{what}: O max-abs {self.max_abs:.3e} > {O_MAX_ABS}"
        else:
            res["o_bound_ratio"] = self.ratio
            assert self.ratio <= 1.0, (f"{what}: O error exceeds max(1e-2, 1.125 2^-8 (|O| + A)) by "
                                       f"x{self.ratio:.3f} (max-abs {self.max_abs:.3e})")
        assert rel_rms <= O_REL_RMS, f"{what}: O rel-RMS {rel_rms:.3e} > {O_REL_RMS}"
        assert self.lse_err <= LSE_MAX_ABS, f"{what}: LSE max-abs {self.lse_err:.3e} > {LSE_MAX_ABS}"
        return res


def check(o_gpu: np.ndarray, l_gpu: np.ndarray, o_ref: np.ndarray, l_ref: np.ndarray, what: str = "",
          strict: bool = True, o_abs: np.ndarray = None):
    """Assert the acceptance tolerances on one set of rows; return a dict of the measured errors.
    ``strict=False`` applies the derived per-element bound and needs ``o_abs`` (the oracle's
    attention over |V| for the same rows)."""
    p = Parity(what, strict)
    p.add(o_gpu, l_gpu, o_ref, l_ref, o_abs)
    return p.result()


def prefill_parity_all_rows(x: PrefillInputs, o, lse, what: str, strict: bool = True, alibi_slopes=None,
                            chunk: int = 1 << 16) -> dict:
    """Compare every output row of a prefill with the oracle, ``chunk`` rows at a time."""
    orc = PrefillOracle(x, alibi_slopes)
    oh, lh = host_outputs(o, lse)
    rows = oracle.all_rows(x.len_q, x.case.Hq)
    p = Parity(what, strict)
    for s in range(0, len(rows), chunk):
        r = rows[s:s + chunk]
        go, gl = gather_prefill_rows(x, oh, lh, r)
        ro, rl = orc.rows(r)
        oa = None if strict else orc.rows(r, abs_v=True)[0]
        p.add(go, gl, ro, rl, oa)
    return p.result()


def gpu_decode(x: DecodeInputs, dev="cuda", num_splits=0, with_host_lens=True, window=None):
    import flashattention_forward_fa_gb300 as fa
    c = x.case
    lens = torch.tensor(x.lens, dtype=torch.int32, device=dev)
    o, lse = fa.fa_decode(x.q.to(dev), x.k_cache.to(dev), x.v_cache.to(dev), lens,
                          window=c.window if window is None else window, scale=c.softmax_scale,
                          num_splits=num_splits, seqlens_k_host=x.lens if with_host_lens else None)
    torch.cuda.synchronize()
    return o, lse


def oracle_decode_rows(x: DecodeInputs, rows: np.ndarray, window=None, abs_v: bool = False):
    """rows: (b, h) pairs.  The decode query is row 0 of a 1-row sequence whose keys are
    cache slots 0 .. len-1; with bottom-right causal alignment it sees every one of them."""
    c = x.case
    q4 = x.q.reshape(c.B, 1, c.Hq, c.d)
    trip = np.zeros((len(rows), 3), dtype=np.int32)
    trip[:, 0] = rows[:, 0]
    trip[:, 1] = rows[:, 1]
    vb = bf16_bits(x.v_cache)
    return oracle.attention_rows(bf16_bits(q4), bf16_bits(x.k_cache), abs_bits(vb) if abs_v else vb,
                                 list(range(c.B)), [1] * c.B, [b * c.Ncap for b in range(c.B)], x.lens,
                                 c.softmax_scale, True, c.window if window is None else window, trip)
