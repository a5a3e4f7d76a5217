"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself: a brute-force loop
written separately here, torch's float64 CPU scaled_dot_product_attention (a
library routine for the special cases it covers), closed forms, and
invariants of the definition.  A final test plants plausible mistakes in
wrappers around the oracle and checks that some pin catches each one.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import ref_numpy
from fa_workloads import bf16_bits

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------- helpers

def to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def c_oracle_seq(q, k, v, scale, causal=False, window=0):
    """C oracle on one sequence given bf16 tensors q [lq,Hq,d], k/v [lk,Hkv,d]."""
    lq, hq, d = q.shape
    lk = k.shape[0]
    rows = oracle.all_rows([lq], hq)
    o, lse = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v),
                                   [0], [lq], [0], [lk], scale, causal, window, rows)
    O = np.zeros((lq, hq, d))
    L = np.full((hq, lq), -np.inf)
    for n, (_, h, i) in enumerate(rows):
        O[i, h] = o[n]
        L[h, i] = lse[n]
    return O, L


def np_oracle_seq(q, k, v, scale, causal=False, window=0):
    return ref_numpy.attention(f64(q), f64(k), f64(v), scale, causal, window)


def brute_force(q, k, v, scale, causal=False, window=0):
    """Scalar loops with math.exp; written independently of both oracles."""
    qd, kd, vd = f64(q), f64(k), f64(v)
    lq, hq, d = qd.shape
    lk, hkv, _ = kd.shape
    O = np.zeros((lq, hq, d))
    L = np.full((hq, lq), -np.inf)
    for h in range(hq):
        g = h * hkv // hq
        for i in range(lq):
            pos = i + lk - lq
            keys = []
            for j in range(lk):
                if causal and (j > pos or (window > 0 and pos - j >= window)):
                    continue
                if not causal and window > 0 and abs(pos - j) >= window:
                    continue
                keys.append(j)
            if not keys:
                continue
            sc = [scale * sum(qd[i, h, t] * kd[j, g, t] for t in range(d)) for j in keys]
            m = max(sc)
            w = [math.exp(s - m) for s in sc]
            z = sum(w)
            for t in range(d):
                O[i, h, t] = sum(w[n] * vd[keys[n], g, t] for n in range(len(keys))) / z
            L[h, i] = m + math.log(z)
    return O, L


def sdpa64(q, k, v, scale, causal=False, window=0):
    """torch float64 CPU SDPA with an explicit boolean mask (rows with keys only)."""
    lq, hq, d = q.shape
    lk, hkv, _ = k.shape
    qq = torch.from_numpy(f64(q)).permute(1, 0, 2)
    kk = torch.from_numpy(f64(k)).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    vv = torch.from_numpy(f64(v)).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    mask = torch.from_numpy(ref_numpy.visible_mask(lq, lk, causal, window))
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
    return out.permute(1, 0, 2).numpy(), mask.any(dim=1).numpy()


def rand_seq(lq, lk, hq, hkv, d, kmult=1.0):
    q = to_bf16(RNG.standard_normal((lq, hq, d)))
    k = to_bf16(RNG.standard_normal((lk, hkv, d)) * kmult)
    v = to_bf16(RNG.standard_normal((lk, hkv, d)))
    return q, k, v


MODES = [
    # lq, lk, hq, hkv, d, causal, window
    (7, 7, 2, 2, 8, False, 0),
    (5, 9, 4, 2, 8, False, 0),
    (9, 5, 2, 1, 4, True, 0),      # Nq > Nk: first rows fully masked
    (6, 11, 4, 1, 8, True, 0),     # Nq < Nk, MQA
    (12, 12, 3, 3, 4, True, 3),    # causal window
    (8, 13, 2, 2, 4, False, 4),    # non-causal window
    (10, 10, 6, 2, 16, True, 1),   # window 1 = diagonal only
]


# ----------------------------------------------------------------------------- cross-checks

@pytest.mark.parametrize("mode", MODES)
def test_c_numpy_bruteforce_sdpa_agree(mode):
    lq, lk, hq, hkv, d, causal, window = mode
    q, k, v = rand_seq(lq, lk, hq, hkv, d, kmult=1.5)
    scale = 1.0 / math.sqrt(d)
    Oc, Lc = c_oracle_seq(q, k, v, scale, causal, window)
    On, Ln = np_oracle_seq(q, k, v, scale, causal, window)
    Ob, Lb = brute_force(q, k, v, scale, causal, window)
    np.testing.assert_allclose(Oc, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(On, Ob, rtol=0, atol=1e-12)
    assert np.array_equal(np.isinf(Lc), np.isinf(Lb)) and np.array_equal(np.isinf(Ln), np.isinf(Lb))
    fin = np.isfinite(Lb)
    np.testing.assert_allclose(Lc[fin], Lb[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(Ln[fin], Lb[fin], rtol=0, atol=1e-12)
    Os, has = sdpa64(q, k, v, scale, causal, window)
    np.testing.assert_allclose(Oc[has], Os[has], rtol=0, atol=1e-12)
    assert np.all(Oc[~has] == 0.0)


def test_lse_matches_torch_logsumexp():
    q, k, v = rand_seq(6, 10, 2, 2, 8)
    scale = 0.3
    _, L = c_oracle_seq(q, k, v, scale)
    s = torch.einsum("ihd,jhd->hij", torch.from_numpy(f64(q)), torch.from_numpy(f64(k))) * scale
    np.testing.assert_allclose(L, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- closed forms

def test_identical_keys_give_mean_of_values():
    lq, lk, d = 5, 9, 8
    q = to_bf16(RNG.standard_normal((lq, 1, d)))
    krow = RNG.standard_normal((1, 1, d))
    k = to_bf16(np.repeat(krow, lk, axis=0))
    v = to_bf16(RNG.standard_normal((lk, 1, d)))
    scale = 0.25
    O, L = c_oracle_seq(q, k, v, scale)
    vmean = f64(v).mean(axis=0)[0]
    s = scale * f64(q)[:, 0, :] @ f64(k)[0, 0, :]
    for i in range(lq):
        np.testing.assert_allclose(O[i, 0], vmean, atol=1e-12)
        assert abs(L[0, i] - (s[i] + math.log(lk))) < 1e-12


def test_identical_keys_causal_prefix_mean():
    # causal: row i (Nq = Nk) averages v_0..v_i and LSE = s + ln(i+1)
    n, d = 6, 4
    q = to_bf16(RNG.standard_normal((n, 1, d)))
    k = to_bf16(np.repeat(RNG.standard_normal((1, 1, d)), n, axis=0))
    v = to_bf16(RNG.standard_normal((n, 1, d)))
    O, L = c_oracle_seq(q, k, v, 1.0, causal=True)
    s = f64(q)[:, 0, :] @ f64(k)[0, 0, :]
    for i in range(n):
        np.testing.assert_allclose(O[i, 0], f64(v)[: i + 1, 0].mean(axis=0), atol=1e-12)
        assert abs(L[0, i] - (s[i] + math.log(i + 1))) < 1e-12


def test_rows_sum_to_one():
    # V = 1 everywhere => every row with at least one key returns exactly 1
    for lq, lk, causal, window in [(7, 7, False, 0), (9, 5, True, 0), (8, 12, True, 3), (8, 12, False, 2)]:
        q, k, _ = rand_seq(lq, lk, 2, 2, 8, kmult=3.0)
        v = to_bf16(np.ones((lk, 2, 8)))
        O, L = c_oracle_seq(q, k, v, 0.5, causal, window)
        has = np.isfinite(L).T   # [lq, hq]
        np.testing.assert_allclose(O[has], 1.0, atol=1e-12)
        assert np.all(O[~has] == 0.0)


def test_causal_row0_is_v0():
    n, d = 8, 8
    q, k, v = rand_seq(n, n, 2, 2, d)
    O, L = c_oracle_seq(q, k, v, 0.7, causal=True)
    for h in range(2):
        np.testing.assert_allclose(O[0, h], f64(v)[0, h], atol=1e-15)
        assert abs(L[h, 0] - 0.7 * float(f64(q)[0, h] @ f64(k)[0, h])) < 1e-12


def test_window_one_returns_diagonal_value():
    lq, lk, d = 6, 10, 8
    q, k, v = rand_seq(lq, lk, 4, 2, d)
    O, L = c_oracle_seq(q, k, v, 0.3, causal=True, window=1)
    for h in range(4):
        g = h // 2
        for i in range(lq):
            p = i + lk - lq
            np.testing.assert_allclose(O[i, h], f64(v)[p, g], atol=1e-15)
            assert abs(L[h, i] - 0.3 * float(f64(q)[i, h] @ f64(k)[p, g])) < 1e-12


def test_zero_query_gives_uniform_weights():
    lk = 11
    q = to_bf16(np.zeros((3, 1, 1)))
    k = to_bf16(RNG.standard_normal((lk, 1, 1)))
    v = to_bf16(RNG.standard_normal((lk, 1, 1)))
    O, L = c_oracle_seq(q, k, v, 5.0)
    np.testing.assert_allclose(O[:, 0, 0], f64(v)[:, 0, 0].mean(), atol=1e-12)
    np.testing.assert_allclose(L, math.log(lk), atol=1e-12)


def test_two_key_softmax_by_hand():
    # q = e0, k0 = e0, k1 = e1, scale 2: s = (2, 0), p0 = 1/(1+e^-2)
    q = to_bf16(np.array([[[1.0, 0.0]]]))
    k = to_bf16(np.array([[[1.0, 0.0]], [[0.0, 1.0]]]))
    v = to_bf16(np.array([[[3.0, -1.0]], [[-5.0, 2.0]]]))
    O, L = c_oracle_seq(q, k, v, 2.0)
    p0 = 1.0 / (1.0 + math.exp(-2.0))
    np.testing.assert_allclose(O[0, 0], [3.0 * p0 - 5.0 * (1 - p0), -p0 + 2.0 * (1 - p0)], atol=1e-14)
    assert abs(L[0, 0] - math.log(math.exp(2.0) + 1.0)) < 1e-14


def test_one_hot_keys_large_scale_select_argmax():
    d = 8
    k = to_bf16(np.eye(d)[:, None, :])          # key j = e_j
    v = to_bf16(RNG.standard_normal((d, 1, d)))
    q = to_bf16(np.eye(d)[[3, 5, 0], None, :])  # query picks key 3, 5, 0
    O, _ = c_oracle_seq(q, k, v, 100.0)
    for r, j in enumerate([3, 5, 0]):
        np.testing.assert_allclose(O[r, 0], f64(v)[j, 0], atol=1e-12)


def test_fully_masked_rows_are_zero_with_neg_inf_lse():
    q, k, v = rand_seq(9, 4, 2, 2, 4)
    O, L = c_oracle_seq(q, k, v, 1.0, causal=True)   # rows 0..4 see no key
    assert np.all(O[:5] == 0.0) and np.all(np.isneginf(L[:, :5]))
    assert np.all(np.isfinite(L[:, 5:]))
    # empty key set
    rows = np.array([[0, 0, 0], [0, 1, 2]], dtype=np.int32)
    o, lse = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), [0], [9], [0], [0],
                                   1.0, False, 0, rows)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))


# ----------------------------------------------------------------------------- invariants

def test_gqa_equals_mha_with_repeated_kv():
    q, k, v = rand_seq(7, 9, 8, 2, 8)
    krep = k.repeat_interleave(4, dim=1)
    vrep = v.repeat_interleave(4, dim=1)
    for causal, window in [(False, 0), (True, 0), (True, 4)]:
        O1, L1 = c_oracle_seq(q, k, v, 0.4, causal, window)
        O2, L2 = c_oracle_seq(q, krep, vrep, 0.4, causal, window)
        np.testing.assert_array_equal(O1, O2)
        np.testing.assert_array_equal(L1, L2)


def test_packed_varlen_equals_per_sequence():
    lens_q, lens_k = [5, 1, 8], [7, 3, 8]
    hq, hkv, d = 4, 2, 8
    seqs = [rand_seq(a, b, hq, hkv, d) for a, b in zip(lens_q, lens_k)]
    Q = torch.cat([s[0] for s in seqs]); K = torch.cat([s[1] for s in seqs]); V = torch.cat([s[2] for s in seqs])
    qo = np.concatenate([[0], np.cumsum(lens_q)[:-1]]); ko = np.concatenate([[0], np.cumsum(lens_k)[:-1]])
    rows = oracle.all_rows(lens_q, hq)
    for causal in (False, True):
        o, lse = oracle.attention_rows(bf16_bits(Q), bf16_bits(K), bf16_bits(V), qo, lens_q, ko, lens_k,
                                       0.5, causal, 0, rows)
        for n, (b, h, i) in enumerate(rows):
            Ob, Lb = c_oracle_seq(*seqs[b], 0.5, causal)
            np.testing.assert_array_equal(o[n], Ob[i, h])
            assert lse[n] == Lb[h, i]


def test_key_permutation_invariance_noncausal():
    q, k, v = rand_seq(5, 12, 2, 2, 8)
    perm = torch.from_numpy(RNG.permutation(12))
    O1, L1 = c_oracle_seq(q, k, v, 0.6)
    O2, L2 = c_oracle_seq(q, k[perm], v[perm], 0.6)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)


@pytest.mark.parametrize("cuts", [[4], [1, 6], [0, 10], [3, 3, 7]])
def test_split_merge_identity(cuts):
    # decode: one query over lk keys, split into chunks and merged back
    lk, hq, hkv, d = 10, 4, 2, 8
    q, k, v = rand_seq(1, lk, hq, hkv, d, kmult=2.0)
    O, L = np_oracle_seq(q, k, v, 0.35)
    bounds = [0] + cuts + [lk]
    parts_o, parts_l = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b > a:
            Oi, Li = np_oracle_seq(q, k[a:b], v[a:b], 0.35)
        else:   # empty chunk: no key
            Oi, Li = np.zeros((1, hq, d)), np.full((hq, 1), -np.inf)
        parts_o.append(Oi[0])   # [hq, d]
        parts_l.append(Li[:, 0])
    Om, Lm = ref_numpy.merge_partials(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(Om, O[0], atol=1e-12)
    np.testing.assert_allclose(Lm, L[:, 0], atol=1e-12)


def test_merge_all_empty_is_zero():
    Om, Lm = ref_numpy.merge_partials(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(Om == 0.0) and np.all(np.isneginf(Lm))


def test_padded_equals_truncated():
    # padded layout: sequence b uses only its first len rows of an N-row slot
    B, N, hq, d = 2, 9, 2, 4
    q, k, v = rand_seq(B * N, B * N, hq, hq, d)
    lens = [4, 9]
    offs = [0, N]
    rows = oracle.all_rows(lens, hq)
    o, lse = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), offs, lens, offs, lens,
                                   0.5, True, 0, rows)
    for n, (b, h, i) in enumerate(rows):
        sl = slice(offs[b], offs[b] + lens[b])
        Ob, Lb = c_oracle_seq(q[sl], k[sl], v[sl], 0.5, True)
        np.testing.assert_array_equal(o[n], Ob[i, h])


# ----------------------------------------------------------------------------- planted mistakes

def _pins(fn) -> list:
    """Run a battery of pins against an oracle-like fn(q,k,v,scale,causal,window)->(O,L)."""
    failed = []
    for mode in MODES:
        lq, lk, hq, hkv, d, causal, window = mode
        rs = np.random.default_rng(7)
        q = to_bf16(rs.standard_normal((lq, hq, d)))
        k = to_bf16(rs.standard_normal((lk, hkv, d)) * 1.5)
        v = to_bf16(rs.standard_normal((lk, hkv, d)))
        O, L = fn(q, k, v, 1.0 / math.sqrt(d), causal, window)
        Ob, Lb = brute_force(q, k, v, 1.0 / math.sqrt(d), causal, window)
        fin = np.isfinite(Lb)
        if (not np.allclose(O, Ob, atol=1e-9) or not np.array_equal(np.isfinite(L), fin)
                or not np.allclose(L[fin], Lb[fin], atol=1e-9)):
            failed.append(mode)
    return failed


def test_pins_pass_for_oracle():
    assert _pins(c_oracle_seq) == []
    assert _pins(np_oracle_seq) == []


MUTANTS = {
    "scale dropped": lambda q, k, v, s, c, w: c_oracle_seq(q, k, v, 1.0, c, w),
    "causal off by one": lambda q, k, v, s, c, w: (
        c_oracle_seq(q, k[:-1], v[:-1], s, c, w) if c and k.shape[0] > 1 else c_oracle_seq(q, k, v, s, c, w)),
    "top-left causal alignment": lambda q, k, v, s, c, w: (
        c_oracle_seq(q, k[: q.shape[0]], v[: q.shape[0]], s, c, w) if c and k.shape[0] > q.shape[0]
        else c_oracle_seq(q, k, v, s, c, w)),
    "window ignored": lambda q, k, v, s, c, w: c_oracle_seq(q, k, v, s, c, 0),
    "wrong GQA map (h % Hkv)": lambda q, k, v, s, c, w: c_oracle_seq(
        q, k[:, [h % k.shape[1] for h in range(q.shape[1])]], v[:, [h % k.shape[1] for h in range(q.shape[1])]], s, c, w),
    "K and V swapped": lambda q, k, v, s, c, w: c_oracle_seq(q, v, k, s, c, w),
    "no max subtraction bug (lse off by max)": lambda q, k, v, s, c, w: (
        lambda r: (r[0], np.where(np.isfinite(r[1]), r[1] - 1e-3, r[1])))(c_oracle_seq(q, k, v, s, c, w)),
    "negated scores": lambda q, k, v, s, c, w: c_oracle_seq(q, k, v, -s, c, w),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistakes_are_caught(name):
    assert _pins(MUTANTS[name]) != [], f"pins did not catch: {name}"


# ----------------------------------------------------------------------------- ALiBi

def brute_force_alibi(q, k, v, scale, causal, window, slopes):
    """Scalar loops: score = scale q.k - m_h |p - j|, p = i + lk - lq (written independently)."""
    qd, kd, vd = f64(q), f64(k), f64(v)
    lq, hq, d = qd.shape
    lk, hkv, _ = kd.shape
    O = np.zeros((lq, hq, d))
    L = np.full((hq, lq), -np.inf)
    for h in range(hq):
        g = h * hkv // hq
        for i in range(lq):
            pos = i + lk - lq
            keys = [j for j in range(lk)
                    if not (causal and (j > pos or (window > 0 and pos - j >= window)))
                    and not (not causal and window > 0 and abs(pos - j) >= window)]
            if not keys:
                continue
            sc = [scale * sum(qd[i, h, t] * kd[j, g, t] for t in range(d)) - slopes[h] * abs(pos - j) for j in keys]
            m = max(sc)
            w = [math.exp(s - m) for s in sc]
            z = sum(w)
            for t in range(d):
                O[i, h, t] = sum(w[n] * vd[keys[n], g, t] for n in range(len(keys))) / z
            L[h, i] = m + math.log(z)
    return O, L


def c_oracle_alibi(q, k, v, scale, causal, window, slopes):
    lq, hq, d = q.shape
    rows = oracle.all_rows([lq], hq)
    o, lse = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), [0], [lq], [0], [k.shape[0]],
                                   scale, causal, window, rows, alibi_slopes=slopes)
    O = np.zeros((lq, hq, d))
    L = np.full((hq, lq), -np.inf)
    for n, (_, h, i) in enumerate(rows):
        O[i, h] = o[n]
        L[h, i] = lse[n]
    return O, L


@pytest.mark.parametrize("mode", MODES)
def test_alibi_c_numpy_bruteforce_agree(mode):
    lq, lk, hq, hkv, d, causal, window = mode
    q, k, v = rand_seq(lq, lk, hq, hkv, d)
    slopes = np.array([0.5 ** (h + 1) for h in range(hq)])
    Oc, Lc = c_oracle_alibi(q, k, v, 0.4, causal, window, slopes)
    On, Ln = ref_numpy.attention(f64(q), f64(k), f64(v), 0.4, causal, window, alibi_slopes=slopes)
    Ob, Lb = brute_force_alibi(q, k, v, 0.4, causal, window, slopes)
    fin = np.isfinite(Lb)
    for O, L in ((Oc, Lc), (On, Ln)):
        np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
        assert np.array_equal(np.isfinite(L), fin)
        np.testing.assert_allclose(L[fin], Lb[fin], rtol=0, atol=1e-12)


def test_alibi_zero_query_gives_geometric_weights():
    # q = 0, causal, Nq = Nk: row i weights key j by r^(i - j), r = exp(-m)
    n, d, m = 9, 4, 0.7
    q = to_bf16(np.zeros((n, 1, d)))
    k = to_bf16(RNG.standard_normal((n, 1, d)))
    v = to_bf16(RNG.standard_normal((n, 1, d)))
    O, L = c_oracle_alibi(q, k, v, 1.0, True, 0, np.array([m]))
    r = math.exp(-m)
    for i in range(n):
        w = np.array([r ** (i - j) for j in range(i + 1)])
        np.testing.assert_allclose(O[i, 0], (w[:, None] * f64(v)[: i + 1, 0]).sum(0) / w.sum(), atol=1e-12)
        assert abs(L[0, i] - math.log((1 - r ** (i + 1)) / (1 - r))) < 1e-12


def test_alibi_zero_slope_is_plain_attention():
    q, k, v = rand_seq(6, 11, 4, 2, 8)
    for causal in (False, True):
        O1, L1 = c_oracle_alibi(q, k, v, 0.3, causal, 0, np.zeros(4))
        O2, L2 = c_oracle_seq(q, k, v, 0.3, causal, 0)
        np.testing.assert_array_equal(O1, O2)
        np.testing.assert_array_equal(L1, L2)


def test_alibi_sign_mistake_is_caught():
    q, k, v = rand_seq(5, 8, 2, 2, 4)
    slopes = np.array([0.25, 0.5])
    Ob, Lb = brute_force_alibi(q, k, v, 0.5, True, 0, slopes)
    Om, Lm = c_oracle_alibi(q, k, v, 0.5, True, 0, -slopes)    # planted: bias added with the wrong sign
    assert not np.allclose(Om, Ob, atol=1e-6)


# ----------------------------------------------------------------------------- RoPE

from oracle import rope as orope  # noqa: E402


def test_rope_tables_match_math():
    c, s = orope.tables(50, 16, base=10000.0)
    for p in (0, 1, 7, 49):
        for i in range(8):
            ang = p * 10000.0 ** (-2.0 * i / 16)
            assert abs(c[p, i] - math.cos(ang)) < 1e-15 and abs(s[p, i] - math.sin(ang)) < 1e-15


def test_rope_rotation_against_scalar_loop():
    x = RNG.standard_normal((6, 3, 12))
    pos = [0, 5, 2, 9, 1, 3]
    c, s = orope.tables(10, 8)
    r = orope.rotate(x, pos, c, s, 8)
    for n in range(6):
        for h in range(3):
            for i in range(4):
                a, b = x[n, h, 2 * i], x[n, h, 2 * i + 1]
                cc, ss = c[pos[n], i], s[pos[n], i]
                assert abs(r[n, h, 2 * i] - (a * cc - b * ss)) < 1e-14
                assert abs(r[n, h, 2 * i + 1] - (a * ss + b * cc)) < 1e-14
            np.testing.assert_array_equal(r[n, h, 8:], x[n, h, 8:])   # past rotary_dim: unchanged


def test_rope_position_zero_is_identity_and_norms_kept():
    x = RNG.standard_normal((5, 2, 16))
    c, s = orope.tables(8, 16)
    np.testing.assert_allclose(orope.rotate(x, [0] * 5, c, s, 16), x, atol=1e-15)
    r = orope.rotate(x, [1, 2, 3, 4, 7], c, s, 16)
    np.testing.assert_allclose((r ** 2).sum(-1), (x ** 2).sum(-1), rtol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    # <R(m) q, R(n) k> is unchanged when every position moves by the same shift
    q = RNG.standard_normal((7, 1, 16))
    k = RNG.standard_normal((7, 1, 16))
    c, s = orope.tables(64, 16)
    pos = np.arange(7)
    s0 = orope.rotate(q, pos, c, s, 16)[:, 0] @ orope.rotate(k, pos, c, s, 16)[:, 0].T
    s1 = orope.rotate(q, pos + 40, c, s, 16)[:, 0] @ orope.rotate(k, pos + 40, c, s, 16)[:, 0].T
    np.testing.assert_allclose(s0, s1, atol=1e-12)
    # and a planted mistake (pairing dimension i with i + d/2 while the tables assume
    # adjacent pairs) is not a rotation of adjacent pairs: position 1 differs
    x = RNG.standard_normal((1, 1, 16))
    r_adj = orope.rotate(x, [1], c, s, 16)
    half = np.concatenate([x[..., 0::2], x[..., 1::2]], axis=-1)
    assert not np.allclose(r_adj, orope.rotate(half, [1], c, s, 16))


def _bf16_bits_of(v):
    """The bf16 pattern of a float64 value that is exactly a bf16 number (its float32 upper half)."""
    w = np.array([v], dtype=np.float32).view(np.uint32)[0]
    assert (w & 0xFFFF) == 0, "not a bf16 value"
    return int(w >> 16)


def test_bf16_rounding_ties_neighbours_zeros():
    # Worked from the format: near 1.0 the bf16 spacing is 2^-7 (1.0 = 0x3F80, next 0x3F81 = 1 + 2^-7).
    r = orope.bf16_round_bits
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),                  # a tie between 0x3F80 and 0x3F81: the even pattern
        (1.0 + 3 * 2.0 ** -8, 0x3F82),              # a tie between 0x3F81 and 0x3F82: the even pattern
        (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),     # just above a tie: up
        (1.0 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),     # just below a tie: down
        # above a tie by less than half a float32 ulp: rounding through float32 would first land on
        # the tie and then go down to 0x3F80; one rounding of the float64 value goes up
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),
        (-(1.0 + 2.0 ** -8), 0xBF80),
        (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),                      # smallest subnormal
        (2.0 ** -134, 0x0000),                      # half of it: a tie with zero, which is even
        (3 * 2.0 ** -135, 0x0001),                  # above that tie
        (3 * 2.0 ** -134, 0x0002),                  # a tie between 0x0001 and 0x0002: even
        (2.0 ** -126 - 2.0 ** -140, 0x0080),        # rounds up onto the smallest normal
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),     # largest finite
        ((2 - 2.0 ** -8) * 2.0 ** 127 - 2.0 ** 100, 0x7F7F),
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),     # the midpoint to 2^128 is a tie: even = infinity
        (-3.0e39, 0xFF80),
        (math.pi, 0x4049),                          # 3.140625 = 0x4049 is nearest to pi
    ]
    got = r(np.array([c[0] for c in cases]))
    for (x, want), g in zip(cases, got):
        assert int(g) == want, f"{x!r}: 0x{int(g):04X} != 0x{want:04X}"
    nan = int(orope.bf16_round_bits(np.nan))
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x007F) != 0      # NaN stays NaN


def test_bf16_rounding_is_the_nearest_bf16_value():
    # Brute force over the format: list every finite non-negative bf16 value in order and pick, for
    # each sample, the nearer of its two neighbours (on a tie, the one with the even pattern).
    pats = np.arange(0x0000, 0x7F80, dtype=np.uint32)
    vals = (pats << np.uint32(16)).view(np.float32).astype(np.float64)
    assert np.all(np.diff(vals) > 0)
    rng = np.random.default_rng(77)
    mags = np.concatenate([
        rng.standard_normal(20000) * 4,
        np.exp(rng.uniform(-95, 88, 20000)),                        # the whole exponent range
        vals[rng.integers(0, len(vals), 5000)],                     # exact bf16 values
        0.5 * (vals[:-1] + vals[1:])[rng.integers(0, len(vals) - 1, 5000)],   # exact midpoints (ties)
    ])
    xs = np.concatenate([mags, -mags])
    a = np.abs(xs)
    hi = np.searchsorted(vals, a, side="left")          # vals[hi - 1] < a <= vals[hi]
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    exact = vals[hi] == a
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick_hi = exact | (dhi < dlo) | ((dhi == dlo) & (pats[hi] % 2 == 0))
    want = np.where(pick_hi, pats[hi], pats[lo]).astype(np.uint32)
    want = want | (np.signbit(xs).astype(np.uint32) << np.uint32(15))
    got = orope.bf16_round_bits(xs).astype(np.uint32)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, e.g. {xs[bad[0]]!r}: 0x{got[bad[0]]:04X} vs 0x{want[bad[0]]:04X}"


def test_rotate_bf16_rounds_the_fp64_rotation_once():
    # rotate_bf16 = one RNE rounding of the fp64 rotation, element by element
    x = torch.from_numpy(RNG.standard_normal((9, 2, 16)).astype(np.float32)).to(torch.bfloat16)
    pos = [0, 1, 2, 3, 5, 8, 13, 21, 34]
    c, s = orope.tables(40, 12)
    exact = orope.rotate(x.to(torch.float64).numpy(), pos, c, s, 12)
    got = orope.rotate_bf16(x, pos, c, s, 12)
    assert got.dtype == torch.bfloat16
    np.testing.assert_array_equal(got.view(torch.int16).numpy().view(np.uint16), orope.bf16_round_bits(exact))
    # every rotated value is within half a bf16 spacing of the fp64 rotation
    g = got.to(torch.float64).numpy()
    _, e = np.frexp(np.abs(exact))
    assert np.all(np.abs(g - exact) <= np.ldexp(1.0, np.maximum(e, -125) - 9))
    np.testing.assert_array_equal(g[..., 12:], x.to(torch.float64).numpy()[..., 12:])


# ------------------------------------------------------------------ stored oracle outputs (regression)

def test_oracle_matches_its_stored_outputs():
    # tests/golden/oracle_small.json was written by tests/golden/make_golden.py from the oracle; a
    # change to the oracle's arithmetic shows up here (and must name the passage that justifies it)
    import json
    import os
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    sys.path.insert(0, os.path.join(here, "golden"))
    import make_golden
    stored = json.load(open(os.path.join(here, "golden", "oracle_small.json")))["cases"]
    fresh = make_golden.build()
    assert [c["name"] for c in stored] == [c["name"] for c in fresh]
    for a, b in zip(stored, fresh):
        np.testing.assert_allclose(b["o"], a["o"], rtol=0, atol=1e-12, err_msg=a["name"])
        np.testing.assert_allclose(b["lse"], a["lse"], rtol=0, atol=1e-12, err_msg=a["name"])
