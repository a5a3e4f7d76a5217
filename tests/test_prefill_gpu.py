"""GPU parity of the prefill kernel against the fp64 oracle (through the C ABI).

Every case compares every output row with the oracle, the full-size named
workloads included (llama7b_causal: 262,144 rows, gqa_window: 524,288 rows,
compared in chunks); a few extra schedules at large sizes compare sampled rows
(tile edges, first/last, random) on top of that.  Tolerances: see tests/_util.py.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from fa_workloads import (BERT_VARLEN, GQA_WINDOW, LLAMA7B_CAUSAL, TINY_MHA, PrefillCase, make_prefill,
                          shrink)
from tests._util import (PrefillOracle, check, gather_prefill_rows, gpu_prefill, oracle_prefill_rows,
                         prefill_parity_all_rows, sample_rows)

pytestmark = pytest.mark.gpu


def _full_parity(case: PrefillCase, strict: bool = True):
    x = make_prefill(case)
    o, lse = gpu_prefill(x)
    res = prefill_parity_all_rows(x, o, lse, case.name, strict=strict)
    import flashattention_forward_fa_gb300 as fa
    assert fa.fa_device_status() == 0
    return x, o, lse, res


# ------------------------------------------------------------------ the named workloads

def test_tiny_mha_full():
    _full_parity(TINY_MHA)


def test_bert_varlen_full():
    _full_parity(BERT_VARLEN)


@pytest.mark.parametrize("case", [LLAMA7B_CAUSAL, GQA_WINDOW], ids=lambda c: c.name)
def test_full_size_every_row(case):
    # the named full-size workloads, launched as the bench launches them, every output row
    # compared with the oracle at the acceptance tolerances
    _, o, lse, res = _full_parity(case)
    assert res["rows"] == case.B * case.Hq * case.Nq and res["empty_rows"] == 0
    assert res["o_loose_elems"] == 0


@pytest.mark.parametrize("case", [
    # one long MQA sequence: 128 items, each walking up to 256 K/V tiles
    PrefillCase("long_context_32k_mqa", B=1, Hq=4, Hkv=1, Nq=32768, Nk=32768, d=128, causal=True, seed=21),
    # d=64 GQA with a ragged tail: 384 items, three snake rounds per resident CTA
    PrefillCase("d64_gqa_three_rounds", B=2, Hq=16, Hkv=4, Nq=3000, Nk=3000, d=64, causal=True, seed=22),
    # non-causal at the persistent grid: every item walks every K/V tile
    PrefillCase("noncausal_persistent", B=3, Hq=24, Hkv=8, Nq=1100, Nk=1700, d=128, seed=23),
], ids=lambda c: c.name)
def test_persistent_schedules_sampled(case):
    x = make_prefill(case)
    o, lse = gpu_prefill(x)
    rows = sample_rows(x, per_head=16, seed=case.seed)
    go, gl = gather_prefill_rows(x, o, lse, rows)
    ro, rl = oracle_prefill_rows(x, rows)
    check(go, gl, ro, rl, case.name)
    assert torch.isfinite(o.float()).all()
    import flashattention_forward_fa_gb300 as fa
    assert fa.fa_device_status() == 0


# ------------------------------------------------------------------ reduced-size families

@pytest.mark.parametrize("case", [
    shrink(LLAMA7B_CAUSAL, name="llama_causal_1k", Hq=4, Hkv=4, Nq=1024, Nk=1024),
    shrink(GQA_WINDOW, name="gqa_window_small", B=2, Hq=8, Hkv=2, Nq=1000, Nk=1000, window=300),
], ids=lambda c: c.name)
def test_reduced_families_full(case):
    _full_parity(case)


# ------------------------------------------------------------------ edge grid

EDGE = []
for d in (64, 128):
    for n in (1, 63, 65, 127, 129, 1000):
        EDGE.append(PrefillCase(f"len{n}_d{d}", B=2, Hq=2, Hkv=2, Nq=n, Nk=n, d=d, seed=100 + n))
        EDGE.append(PrefillCase(f"len{n}_d{d}_causal", B=1, Hq=2, Hkv=1, Nq=n, Nk=n, d=d, causal=True,
                                seed=200 + n))
EDGE += [
    # causal with Nq != Nk, both directions (bottom-right alignment; Nq > Nk fully masks leading rows)
    PrefillCase("causal_q_lt_k", B=2, Hq=4, Hkv=2, Nq=200, Nk=333, d=128, causal=True, seed=301),
    PrefillCase("causal_q_gt_k", B=2, Hq=4, Hkv=2, Nq=333, Nk=200, d=128, causal=True, seed=302),
    PrefillCase("causal_q_gt_k_d64", B=1, Hq=2, Hkv=2, Nq=300, Nk=40, d=64, causal=True, seed=303),
    # noncausal Nq != Nk
    PrefillCase("noncausal_q_ne_k", B=3, Hq=3, Hkv=1, Nq=77, Nk=301, d=64, seed=304),
    # MQA and GQA
    PrefillCase("mqa_h32_kv1", B=1, Hq=32, Hkv=1, Nq=257, Nk=257, d=128, causal=True, seed=305),
    PrefillCase("gqa_h8_kv4", B=2, Hq=8, Hkv=4, Nq=190, Nk=190, d=64, seed=306),
    # windows: 1 (diagonal only), 17, >= N (equals plain causal), non-causal symmetric
    PrefillCase("window1", B=1, Hq=2, Hkv=2, Nq=300, Nk=300, d=128, causal=True, window=1, seed=307),
    PrefillCase("window17", B=1, Hq=2, Hkv=2, Nq=300, Nk=300, d=64, causal=True, window=17, seed=308),
    PrefillCase("window_ge_n", B=1, Hq=2, Hkv=2, Nq=300, Nk=300, d=128, causal=True, window=5000, seed=309),
    PrefillCase("window_noncausal", B=1, Hq=2, Hkv=1, Nq=260, Nk=400, d=64, window=50, seed=310),
    PrefillCase("window_q_lt_k", B=1, Hq=2, Hkv=2, Nq=100, Nk=700, d=128, causal=True, window=200, seed=311),
    # large scores: K drawn x4 sharpens the softmax (exercises the lazy rescale)
    PrefillCase("sharp_scores", B=1, Hq=2, Hkv=2, Nq=700, Nk=700, d=128, causal=True, k_mult=4.0, seed=312),
    PrefillCase("sharp_noncausal", B=1, Hq=2, Hkv=2, Nq=200, Nk=900, d=64, k_mult=4.0, seed=313),
    # packed varlen: one long and many short sequences, an empty sequence, different q/k lengths
    PrefillCase("varlen_long_short", B=6, Hq=4, Hkv=2, Nq=700, Nk=700, d=128, layout="packed",
                len_q=[700, 3, 1, 17, 129, 64], seed=314),
    PrefillCase("varlen_with_empty", B=4, Hq=2, Hkv=2, Nq=300, Nk=300, d=64, layout="packed",
                len_q=[5, 0, 300, 129], len_k=[7, 9, 300, 0], seed=315),
    PrefillCase("varlen_causal_qk", B=3, Hq=4, Hkv=1, Nq=400, Nk=500, d=128, layout="packed", causal=True,
                len_q=[100, 400, 33], len_k=[250, 400, 500], seed=316),
    PrefillCase("varlen_window", B=3, Hq=2, Hkv=2, Nq=600, Nk=600, d=64, layout="packed", causal=True,
                window=64, len_q=[600, 1, 257], seed=317),
    # padded layout with valid lengths (seqlens), including a zero-length sequence
    PrefillCase("padded_seqlens", B=4, Hq=2, Hkv=2, Nq=256, Nk=256, d=128, layout="padded",
                len_q=[256, 100, 0, 129], len_k=[256, 77, 10, 0], seed=318),
    PrefillCase("padded_causal", B=3, Hq=4, Hkv=2, Nq=300, Nk=300, d=64, layout="padded", causal=True,
                len_q=[300, 150, 1], len_k=[300, 200, 7], seed=319),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: c.name)
def test_edge_grid(case):
    # sharpened scores can push |O| past 1.28, where bf16 output rounding alone exceeds 1e-2
    _, o, lse, res = _full_parity(case, strict=case.k_mult <= 2.0)
    if case.layout == "padded":
        # rows past a sequence's valid length are written as zeros with LSE = -inf
        for b, lq in enumerate(case.len_q):
            assert torch.all(o[b, lq:] == 0)
            assert torch.all(torch.isneginf(lse[b, :, lq:]))


def test_zero_length_keys_give_zero_rows():
    case = PrefillCase("no_keys", B=2, Hq=2, Hkv=2, Nq=130, Nk=130, d=64, layout="padded", len_q=[130, 50],
                       len_k=[0, 0], seed=320)
    _, o, lse, res = _full_parity(case)
    assert res["empty_rows"] == 2 * (130 + 50)
    assert torch.all(o == 0)


@pytest.mark.parametrize("d", [64, 128])
def test_nan_in_padding_past_seqlens_k_is_ignored(d):
    # padded layout: K/V rows past a sequence's valid length are in-bounds memory the caller may
    # leave as anything (here NaN and Inf); they must not reach O or the LSE
    import flashattention_forward_fa_gb300 as fa
    case = PrefillCase("nan_padding", B=3, Hq=4, Hkv=2, Nq=200, Nk=300, d=d, layout="padded", causal=True,
                       len_q=[200, 90, 1], len_k=[300, 131, 64], seed=330 + d)
    x = make_prefill(case)
    k, v = x.k.clone(), x.v.clone()
    for b, lk in enumerate(x.len_k):
        k[b, lk:] = float("nan")
        v[b, lk:] = float("nan")
        v[b, lk::3] = float("inf")
    sq = torch.tensor(x.len_q, dtype=torch.int32, device="cuda")
    sk = torch.tensor(x.len_k, dtype=torch.int32, device="cuda")
    o, lse = fa.fa_fwd(x.q.cuda(), k.cuda(), v.cuda(), causal=True, seqlens_q=sq, seqlens_k=sk)
    torch.cuda.synchronize()
    rows = oracle.all_rows(x.len_q, case.Hq)
    go, gl = gather_prefill_rows(x, o, lse, rows)
    ro, rl = oracle_prefill_rows(x, rows)  # the oracle reads only the valid rows of the clean tensors
    check(go, gl, ro, rl, case.name)
    assert torch.isfinite(o.float()).all()
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("d,causal,window,per_key", [(128, True, 0, 0.065), (64, True, 0, 0.065),
                                                      (128, False, 0, 0.065), (64, True, 200, 0.065),
                                                      (128, True, 0, 0.26), (64, False, 0, 0.26),
                                                      (128, True, 300, 0.26), (128, True, 0, 0.42),
                                                      (64, False, 0, 0.42), (128, True, 300, 0.42)],
                         ids=["d128_causal", "d64_causal", "d128_noncausal", "d64_window200", "steep_d128_causal",
                              "steep_d64_noncausal", "steep_d128_window300", "half2_d128_causal",
                              "half2_d64_noncausal", "half2_d128_window300"])
def test_rising_scores_move_the_base(d, causal, window, per_key):
    # Scores that rise along the keys: by ~12 log2 units per 128-key tile (per_key 0.065), so that
    # the weights of a row grow by 2^12 a tile under a fixed exponent base, or by ~48 (per_key
    # 0.26), so that within a few tiles a tile's weights would pass 2^57 and the base must move:
    # the tile's max is taken, O is rescaled and the tile exponentiated again from the scores
    # (on diagonal and window tiles too).  At ~0.6 log2 units per key (per_key 0.42) the first
    # 64 keys of a tile stay below the limit and only the last 64 pass it.  Each row still
    # spreads its weight over a few keys.
    case = PrefillCase(f"rising_d{d}", B=1, Hq=4, Hkv=2, Nq=640, Nk=700, d=d, causal=causal, window=window,
                       seed=340 + d)
    x = make_prefill(case)
    g = torch.Generator().manual_seed(341)
    u = torch.randn(d, generator=g)
    u = u / u.norm()
    a = 4.0                                              # query component along u
    beta = per_key / (case.softmax_scale * a)           # key component per position: per_key nat per key
    ramp = torch.arange(case.Nk, dtype=torch.float32) * beta
    x.q = (x.q.float() + a * u).to(torch.bfloat16)
    x.k = (x.k.float() * 0.25 + ramp[None, :, None, None] * u).to(torch.bfloat16)
    o, lse, _ = _parity_of(x)
    assert torch.isfinite(o.float()).all()


def _parity_of(x):
    import flashattention_forward_fa_gb300 as fa
    o, lse = gpu_prefill(x)
    res = prefill_parity_all_rows(x, o, lse, x.case.name, strict=False)  # |O| ~ |V| > 1.28: derived bound
    assert fa.fa_device_status() == 0
    return o, lse, res


@pytest.mark.parametrize("d,causal,window,rise", [(128, True, 3, [2, 5, 7, 3]), (64, True, 3, [7, 2, 4, 6]),
                                                  (128, True, 40, [3, 6, 2, 7]), (64, False, 20, [5, 2, 7, 4]),
                                                  (128, True, 0, [2, 3, 5, 7])],
                         ids=["d128_w3", "d64_w3", "d128_w40", "d64_noncausal_w20", "d128_causal"])
def test_stale_base_weights_above_one(d, causal, window, rise):
    # The exponent base moves only when a tile's max exceeds it by more than 8 log2 units.  Here
    # every 128-key tile's scores sit 2-7 log2 units above the previous tile's (a per-tile level
    # along one direction u, plus small noise), so a row whose visible keys start in one tile and
    # continue in the next keeps the first tile's base: its largest weights are 2^2 .. 2^7 and are
    # rounded to bf16 like every other weight.  Short windows leave rows a few keys each, so |O|
    # follows single V rows (up to ~4) and the bf16 roundings are at their largest.
    case = PrefillCase(f"stale_base_d{d}", B=1, Hq=4, Hkv=2, Nq=900, Nk=900, d=d, causal=causal,
                       window=window, seed=360 + d + window)
    x = make_prefill(case)
    g = torch.Generator().manual_seed(361 + window)
    u = torch.randn(d, generator=g)
    u = u / u.norm()
    a = 4.0                                                      # query component along u
    lvl = np.concatenate([[0.0], np.cumsum([rise[t % len(rise)] for t in range(8)])])   # log2 units per tile
    key_lvl = torch.tensor(lvl[np.arange(case.Nk) // 128], dtype=torch.float32)
    beta = key_lvl * math.log(2.0) / (case.softmax_scale * a)    # key component along u
    x.q = (x.q.float() * 0.1 + a * u).to(torch.bfloat16)
    x.k = (x.k.float() * 0.1 + beta[None, :, None, None] * u).to(torch.bfloat16)
    o, lse, res = _parity_of(x)
    assert torch.isfinite(o.float()).all()


# ------------------------------------------------------------------ invariances (GPU vs GPU)

def test_varlen_packed_equals_per_sequence_dense():
    import flashattention_forward_fa_gb300 as fa
    case = PrefillCase("v", B=4, Hq=4, Hkv=2, Nq=300, Nk=300, d=128, layout="packed", causal=True,
                       len_q=[300, 17, 129, 64], seed=330)
    x = make_prefill(case)
    o, lse = gpu_prefill(x)
    for b in range(case.B):
        sl = slice(x.q_off[b], x.q_off[b] + x.len_q[b])
        ob, lb = fa.fa_fwd(x.q[sl][None].cuda(), x.k[sl][None].cuda(), x.v[sl][None].cuda(), causal=True)
        assert torch.equal(ob[0], o[sl])
        assert torch.equal(lb[0], lse[:, sl])


def test_gqa_equals_mha_with_repeated_kv():
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(PrefillCase("g", B=2, Hq=8, Hkv=2, Nq=200, Nk=260, d=64, causal=True, seed=331))
    o1, l1 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True)
    krep = x.k.repeat_interleave(4, dim=2).contiguous()
    vrep = x.v.repeat_interleave(4, dim=2).contiguous()
    o2, l2 = fa.fa_fwd(x.q.cuda(), krep.cuda(), vrep.cuda(), causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_window_ge_n_equals_causal():
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(PrefillCase("w", B=1, Hq=2, Hkv=2, Nq=333, Nk=333, d=128, seed=332))
    o1, l1 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True)
    o2, l2 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True, window=333)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_key_permutation_invariance_noncausal():
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(PrefillCase("p", B=1, Hq=2, Hkv=2, Nq=128, Nk=384, d=64, seed=333))
    perm = torch.randperm(384, generator=torch.Generator().manual_seed(0))
    o1, l1 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda())
    o2, l2 = fa.fa_fwd(x.q.cuda(), x.k[:, perm].contiguous().cuda(), x.v[:, perm].contiguous().cuda())
    # summation order changes: compare within the bf16 output tolerance
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_deterministic_repeat():
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(PrefillCase("r", B=1, Hq=4, Hkv=4, Nq=640, Nk=640, d=128, causal=True, seed=334))
    o1, l1 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True)
    o2, l2 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_optional_and_nondefault_stream():
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(PrefillCase("s", B=1, Hq=2, Hkv=2, Nq=256, Nk=256, d=64, seed=335))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), return_lse=False)
    s.synchronize()
    assert l1 is None
    o2, _ = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda())
    assert torch.equal(o1, o2)
