"""The bench's algorithmic-work accounting (the numerator of every roofline fraction) against
closed forms: visible (query, key) pairs under each mask, FLOPs per pair, decode bytes."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from fa_workloads import DECODE_CACHE, GQA_WINDOW, LLAMA7B_CAUSAL, DecodeCase  # noqa: E402


def brute_pairs(lq, lk, causal, window):
    n = 0
    for i in range(lq):
        p = i + lk - lq
        for j in range(lk):
            if causal and j > p:
                continue
            if window > 0 and (p - j >= window or (not causal and j - p >= window)):
                continue
            n += 1
    return n


@pytest.mark.parametrize("lq,lk,causal,window", [
    (7, 7, False, 0), (7, 7, True, 0), (5, 9, True, 0), (9, 5, True, 0), (12, 12, True, 3),
    (12, 12, False, 3), (6, 10, False, 4), (10, 10, True, 1), (1, 50, True, 0), (0, 5, True, 0),
])
def test_visible_pairs_match_brute_force(lq, lk, causal, window):
    assert bench.visible_pairs([lq], [lk], causal, window) == brute_pairs(lq, lk, causal, window)


def test_visible_pairs_closed_forms():
    n = 8192
    assert bench.visible_pairs([n], [n], True, 0) == n * (n + 1) // 2          # causal triangle
    assert bench.visible_pairs([n], [n], False, 0) == n * n
    w = 1024                                                                   # causal window
    assert bench.visible_pairs([4096], [4096], True, w) == sum(min(i + 1, w) for i in range(4096))
    assert bench.visible_pairs([4096], [4096], True, w) == 3_670_528
    assert bench.visible_pairs([3, 4], [3, 4], False, 0) == 9 + 16            # sums over sequences


def test_named_workload_flops():
    c = LLAMA7B_CAUSAL
    assert bench.prefill_flops(c, [c.Nq], [c.Nk]) == 4 * 128 * 32 * 33_558_528 == 549_822_922_752
    g = GQA_WINDOW
    assert bench.prefill_flops(g, [g.Nq] * g.B, [g.Nk] * g.B) == 4 * 128 * 32 * 4 * 3_670_528


def test_decode_bytes_closed_form():
    c = DecodeCase("t", B=3, Hq=8, Hkv=2, Ncap=1000, d=64)
    lens = [10, 0, 1000]
    kv = sum(lens) * 2 * 64 * 2 * 2                 # K and V, bf16, once per KV head
    qo = 2 * 3 * 8 * 64 * 2                         # q in, o out
    assert bench.decode_bytes(c, lens) == kv + qo + 3 * 8 * 4
    w = DecodeCase("w", B=2, Hq=4, Hkv=4, Ncap=500, d=128, window=100)
    assert bench.decode_bytes(w, [50, 400]) == (50 + 100) * 4 * 128 * 4 + 2 * 2 * 4 * 128 * 2 + 2 * 4 * 4
    assert bench.decode_bytes(DECODE_CACHE, [4352] * 64) == 4352 * 64 * 8 * 128 * 4 + 2 * 64 * 32 * 128 * 2 \
        + 64 * 32 * 4
