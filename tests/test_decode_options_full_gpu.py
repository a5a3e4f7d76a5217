"""The decode option rows at full size: decode_cache (B=64, Hq=32, Hkv=8, d=128, cache 8192,
lengths uniform in [512, 8192]) over a paged cache, with four new tokens per sequence, and with
ALiBi, each launched as the bench launches it and compared with the fp64 oracle on every output
row at the acceptance tolerances (paging: the hwcomputing.csdn.net page, §四; several new tokens:
the incremental mode of the agent.csdn.net walkthrough, 结尾, extended to a block of tokens; ALiBi:
the jsqmd page, §三)."""

import numpy as np
import pytest
import torch

import oracle
from fa_workloads import DECODE_CACHE, bf16_bits, make_decode
from tests._util import check, oracle_decode_rows

pytestmark = pytest.mark.gpu


def _pairs(B, Hq):
    return np.array([(b, h) for b in range(B) for h in range(Hq)], dtype=np.int32)


def _check_rows(o, lse, ro, rl, rows, what):
    import flashattention_forward_fa_gb300 as fa
    go = o.float().cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    gl = lse.cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    res = check(go, gl, ro, rl, what)
    assert res["o_loose_elems"] == 0 and res["empty_rows"] == 0
    assert fa.fa_device_status() == 0


def test_paged_decode_cache_full_size_every_row():
    # the cache cut into 128-token pages scattered in a random order through the page pool
    import flashattention_forward_fa_gb300 as fa
    c = DECODE_CACHE
    x = make_decode(c)
    page = 128
    nb = c.Ncap // page
    perm = torch.randperm(c.B * nb, generator=torch.Generator("cpu").manual_seed(61))
    kp = torch.empty((c.B * nb, page, c.Hkv, c.d), dtype=torch.bfloat16)
    vp = torch.empty_like(kp)
    kp[perm] = x.k_cache.reshape(c.B * nb, page, c.Hkv, c.d)
    vp[perm] = x.v_cache.reshape(c.B * nb, page, c.Hkv, c.d)
    table = perm.view(c.B, nb).to(torch.int32).contiguous()
    lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
    o, lse = fa.fa_decode_paged(x.q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens, scale=c.softmax_scale,
                                seqlens_k_host=x.lens)
    torch.cuda.synchronize()
    rows = _pairs(c.B, c.Hq)
    ro, rl = oracle_decode_rows(x, rows)
    _check_rows(o, lse, ro, rl, rows, "paged decode_cache")


def test_alibi_decode_cache_full_size_every_row():
    import flashattention_forward_fa_gb300 as fa
    c = DECODE_CACHE
    x = make_decode(c)
    slopes = np.array(fa.alibi_slopes(c.Hq), dtype=np.float32)
    lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
    o, lse = fa.fa_decode(x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), lens, scale=c.softmax_scale,
                          seqlens_k_host=x.lens, alibi_slopes=slopes)
    torch.cuda.synchronize()
    rows = _pairs(c.B, c.Hq)
    trip = np.zeros((len(rows), 3), dtype=np.int32)
    trip[:, 0], trip[:, 1] = rows[:, 0], rows[:, 1]
    ro, rl = oracle.attention_rows(bf16_bits(x.q.reshape(c.B, 1, c.Hq, c.d)), bf16_bits(x.k_cache),
                                   bf16_bits(x.v_cache), list(range(c.B)), [1] * c.B,
                                   [b * c.Ncap for b in range(c.B)], x.lens, c.softmax_scale, True, 0, trip,
                                   alibi_slopes=slopes.astype(np.float64))
    _check_rows(o, lse, ro, rl, rows, "alibi decode_cache")


def test_four_new_tokens_decode_cache_full_size_every_row():
    # four new tokens per sequence, the last four cache slots (token t sees keys <= len - 4 + t)
    import flashattention_forward_fa_gb300 as fa
    c = DECODE_CACHE
    x = make_decode(c)
    nt = 4
    q = torch.randn(c.B, nt, c.Hq, c.d, generator=torch.Generator("cpu").manual_seed(6)).to(torch.bfloat16)
    lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
    o, lse = fa.fa_decode(q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), lens, scale=c.softmax_scale,
                          seqlens_k_host=x.lens)
    torch.cuda.synchronize()
    rows = oracle.all_rows([nt] * c.B, c.Hq)   # (b, h, t)
    ro, rl = oracle.attention_rows(bf16_bits(q), bf16_bits(x.k_cache), bf16_bits(x.v_cache),
                                   [b * nt for b in range(c.B)], [nt] * c.B, [b * c.Ncap for b in range(c.B)],
                                   x.lens, c.softmax_scale, True, 0, rows)
    # the same tokens through the prefill kernel (padded layout, per-sequence key lengths), as the
    # bench's comparison row runs them
    o2, lse2 = fa.fa_fwd(q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), causal=True, scale=c.softmax_scale,
                         seqlens_k=lens)
    torch.cuda.synchronize()
    for out, l, what in ((o, lse, "decode kernel"), (o2, lse2, "prefill kernel")):
        go = out.float().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]].astype(np.float64)
        gl = l.cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
        res = check(go, gl, ro, rl, "decode_cache, 4 new tokens, " + what)
        assert res["rows"] == c.B * c.Hq * nt and res["o_loose_elems"] == 0
    assert fa.fa_device_status() == 0
