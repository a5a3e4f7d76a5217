"""Decode with several new query tokens per sequence over a KV cache (speculative
decoding, chunked prefill on top of a cache).

The new tokens are the last Nq positions of each sequence: token t of sequence b
sits at position t + len_b - Nq and attends causally to cache slots 0 .. that
position (the incremental mode of the agent.csdn.net walkthrough, 结尾, with the
bottom-right causal alignment).  The library computes this with fa_fwd on the
cache layout: q [B, Nq, Hq, d], k/v = the caches [B, Ncap, Hkv, d], and the
cache lengths as seqlens_k.  Checked against the oracle row by row.
"""

import numpy as np
import pytest
import torch

import oracle
from fa_workloads import bf16_bits
from tests._util import check

pytestmark = pytest.mark.gpu


def _case(B, Nq, Hq, Hkv, Ncap, d, lens, window=0, seed=0):
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, Nq, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Ncap, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Ncap, Hkv, d, generator=g).to(torch.bfloat16)
    return q, k, v, list(lens)


@pytest.mark.parametrize("B,Nq,Hq,Hkv,Ncap,d,lens,window", [
    (4, 4, 8, 2, 1000, 128, [1000, 4, 517, 130], 0),      # speculative decode, 4 draft tokens
    (2, 16, 32, 8, 2048, 128, [2048, 700], 0),            # GQA, 16 new tokens
    (3, 7, 4, 1, 600, 64, [7, 600, 333], 0),              # MQA, d=64, odd token count
    (2, 130, 8, 2, 1500, 128, [1500, 131], 0),            # chunked prefill: chunk spans two Q tiles
    (2, 5, 8, 2, 900, 128, [900, 300], 64),               # sliding window over the cache
])
def test_multitoken_decode_matches_oracle(B, Nq, Hq, Hkv, Ncap, d, lens, window):
    import flashattention_forward_fa_gb300 as fa
    q, k, v, lens = _case(B, Nq, Hq, Hkv, Ncap, d, lens, window, seed=B * 100 + Nq)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, window=window, scale=scale,
                       seqlens_k=lens_dev)
    torch.cuda.synchronize()
    rows = oracle.all_rows([Nq] * B, Hq)
    ro, rl = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), [b * Nq for b in range(B)],
                                   [Nq] * B, [b * Ncap for b in range(B)], lens, scale, True, window, rows)
    go = o.float().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]].astype(np.float64)
    gl = lse.cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
    check(go, gl, ro, rl, f"multitoken B={B} Nq={Nq}")
    assert fa.fa_device_status() == 0


def test_single_token_agrees_with_split_kv_decode():
    # Nq = 1 through the prefill kernel equals the split-KV decode path
    import flashattention_forward_fa_gb300 as fa
    q, k, v, lens = _case(3, 1, 16, 4, 1200, 128, [1200, 65, 640], seed=9)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o1, l1 = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, seqlens_k=lens_dev)
    o2, l2 = fa.fa_decode(q[:, 0].contiguous().cuda(), k.cuda(), v.cuda(), lens_dev, seqlens_k_host=lens)
    assert (o1[:, 0].float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1[:, :, 0] - l2).abs().max().item() <= 1e-3


# ---------------------------------------------------------------- the split-KV decode kernel with Nq new tokens

def _oracle_multitoken(q, k, v, lens, window, scale, alibi=None):
    B, Nq, Hq, d = q.shape
    Ncap = k.shape[1]
    rows = oracle.all_rows([Nq] * B, Hq)
    ro, rl = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), [b * Nq for b in range(B)], [Nq] * B,
                                   [b * Ncap for b in range(B)], lens, scale, True, window, rows,
                                   alibi_slopes=alibi)
    return rows, ro, rl


@pytest.mark.parametrize("B,Nq,Hq,Hkv,Ncap,d,lens,window", [
    (4, 4, 32, 8, 1000, 128, [1000, 4, 517, 130], 0),     # 4 drafts x G=4: one 16-row block
    (2, 16, 32, 8, 2048, 128, [2048, 700], 0),            # 64 rows: four row blocks
    (3, 7, 4, 1, 600, 64, [7, 600, 333], 0),              # MQA, d=64, 28 rows
    (2, 5, 8, 2, 900, 128, [900, 300], 64),               # window: each token its own lower edge
    (3, 6, 8, 8, 500, 128, [3, 0, 400], 0),               # len < Nq: early tokens see nothing
    (2, 3, 16, 1, 1500, 128, [1500, 1401], 100),          # MQA, 48 rows, window
])
def test_decode_kernel_multitoken_matches_oracle(B, Nq, Hq, Hkv, Ncap, d, lens, window):
    import flashattention_forward_fa_gb300 as fa
    q, k, v, lens = _case(B, Nq, Hq, Hkv, Ncap, d, lens, window, seed=B * 77 + Nq + window)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_decode(q.cuda(), k.cuda(), v.cuda(), lens_dev, window=window, scale=scale, seqlens_k_host=lens)
    torch.cuda.synchronize()
    assert o.shape == q.shape and lse.shape == (B, Hq, Nq)
    rows, ro, rl = _oracle_multitoken(q, k, v, lens, window, scale)
    go = o.float().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]].astype(np.float64)
    gl = lse.cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
    check(go, gl, ro, rl, f"decode kernel Nq={Nq}")
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("num_splits", [0, 1, 5])
def test_decode_kernel_multitoken_agrees_with_prefill_path(num_splits):
    import flashattention_forward_fa_gb300 as fa
    q, k, v, lens = _case(3, 4, 16, 4, 1200, 128, [1200, 65, 640], seed=31)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o1, l1 = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, seqlens_k=lens_dev)
    o2, l2 = fa.fa_decode(q.cuda(), k.cuda(), v.cuda(), lens_dev, num_splits=num_splits, seqlens_k_host=lens)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_decode_kernel_multitoken_paged_and_alibi():
    import flashattention_forward_fa_gb300 as fa
    B, Nq, Hq, Hkv, d, page = 3, 4, 16, 4, 128, 64
    lens = [1000, 70, 640]
    q, k, v, _ = _case(B, Nq, Hq, Hkv, 1024, d, lens, seed=32)
    nb = 1024 // page
    g = torch.Generator("cpu").manual_seed(33)
    perm = torch.randperm(B * nb, generator=g)
    kp = torch.empty(B * nb, page, Hkv, d, dtype=torch.bfloat16)
    vp = torch.empty_like(kp)
    kp[perm] = k.reshape(B * nb, page, Hkv, d)
    vp[perm] = v.reshape(B * nb, page, Hkv, d)
    table = perm.reshape(B, nb).to(torch.int32)
    slopes = np.array(fa.alibi_slopes(Hq), np.float32)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / np.sqrt(d)
    for window in (0, 200):
        o, lse = fa.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens_dev, window=window,
                                    scale=scale, seqlens_k_host=lens, alibi_slopes=slopes)
        torch.cuda.synchronize()
        rows, ro, rl = _oracle_multitoken(q, k, v, lens, window, scale, alibi=slopes.astype(np.float64))
        go = o.float().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]].astype(np.float64)
        gl = lse.cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
        check(go, gl, ro, rl, f"paged alibi Nq={Nq} window={window}")
        assert fa.fa_device_status() == 0
