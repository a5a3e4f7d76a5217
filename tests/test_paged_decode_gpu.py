"""Decode over a paged KV cache (block table), against the fp64 oracle.

Each sequence's cache is cut into pages that are scattered in random order
through a larger page pool (the other pool pages hold garbage); the block table
maps logical blocks to pages.  The oracle sees the same keys in their logical
order, so any paging mistake shows as a parity failure.
"""

import numpy as np
import pytest
import torch

import oracle
from fa_workloads import bf16_bits
from tests._util import check

pytestmark = pytest.mark.gpu


def _paged(B, Hq, Hkv, d, lens, page_size, extra_pages=5, seed=0):
    g = torch.Generator("cpu").manual_seed(seed)
    max_blocks = max(1, max((n + page_size - 1) // page_size for n in lens))
    cap = max_blocks * page_size
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, cap, Hkv, d, generator=g).to(torch.bfloat16)   # logical caches
    v = torch.randn(B, cap, Hkv, d, generator=g).to(torch.bfloat16)
    num_pages = B * max_blocks + extra_pages
    perm = torch.randperm(num_pages, generator=g)
    kp = torch.randn(num_pages, page_size, Hkv, d, generator=g).to(torch.bfloat16)  # garbage everywhere
    vp = torch.randn(num_pages, page_size, Hkv, d, generator=g).to(torch.bfloat16)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    n = 0
    for b in range(B):
        for blk in range((lens[b] + page_size - 1) // page_size):
            pg = int(perm[n]); n += 1
            table[b, blk] = pg
            kp[pg] = k[b, blk * page_size:(blk + 1) * page_size]
            vp[pg] = v[b, blk * page_size:(blk + 1) * page_size]
    # unused table entries point at a valid (garbage) page: only keys < len may be read
    table[table < 0] = int(perm[-1])
    return q, k, v, kp, vp, table, cap


@pytest.mark.parametrize("B,Hq,Hkv,d,lens,page_size,window", [
    (4, 16, 4, 128, [1000, 1, 64, 777], 64, 0),
    (3, 8, 2, 128, [2048, 300, 129], 128, 0),
    (2, 32, 8, 128, [4000, 2500], 256, 0),
    (3, 4, 1, 64, [513, 64, 65], 64, 0),          # MQA, d = 64
    (2, 8, 2, 128, [1500, 700], 128, 200),        # window start not on a tile boundary
    (2, 8, 2, 128, [1500, 100], 64, 64),
])
def test_paged_decode_matches_oracle(B, Hq, Hkv, d, lens, page_size, window):
    import flashattention_forward_fa_gb300 as fa
    q, k, v, kp, vp, table, cap = _paged(B, Hq, Hkv, d, lens, page_size, seed=B * 1000 + page_size + window)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens_dev, window=window,
                                scale=scale, seqlens_k_host=lens)
    torch.cuda.synchronize()
    rows = np.array([(b, h, 0) for b in range(B) for h in range(Hq)], dtype=np.int32)
    ro, rl = oracle.attention_rows(bf16_bits(q.reshape(B, 1, Hq, d)), bf16_bits(k), bf16_bits(v),
                                   list(range(B)), [1] * B, [b * cap for b in range(B)], lens, scale, True, window,
                                   rows)
    go = o.float().cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    gl = lse.cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    check(go, gl, ro, rl, f"paged page={page_size}")
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("num_splits", [1, 3, 7])
def test_paged_equals_contiguous_decode(num_splits):
    import flashattention_forward_fa_gb300 as fa
    lens = [1800, 64, 999]
    q, k, v, kp, vp, table, cap = _paged(3, 16, 4, 128, lens, 128, seed=77)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o1, l1 = fa.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens_dev, num_splits=num_splits,
                                seqlens_k_host=lens)
    o2, l2 = fa.fa_decode(q.cuda(), k.cuda(), v.cuda(), lens_dev, num_splits=num_splits, seqlens_k_host=lens)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bad_block_table_entry_is_reported_not_faulted():
    import flashattention_forward_fa_gb300 as fa
    lens = [300, 200]
    q, k, v, kp, vp, table, cap = _paged(2, 8, 2, 128, lens, 64, seed=5)
    table[1, 1] = kp.shape[0] + 1000           # out of range: the kernel must record it and read page 0
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    fa.fa_device_status(clear=True)
    o, lse = fa.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens_dev, seqlens_k_host=lens)
    bits = fa.fa_device_status(clear=True)
    assert bits & 2, "out-of-range page was not reported"
    assert torch.isfinite(o.float()).all()
