"""ALiBi (jsqmd page, §三 "ALiBi位置编码的线性偏置"): every scaled score gets
-m_h |p - j|, p the query's absolute position.  GPU prefill and decode against the
fp64 oracle with the same slopes."""

import numpy as np
import pytest
import torch

import oracle
from fa_workloads import PrefillCase, bf16_bits, make_prefill
from tests._util import check, gather_prefill_rows, oracle_prefill_rows

pytestmark = pytest.mark.gpu


def _slopes(hq):
    import flashattention_forward_fa_gb300 as fa
    return np.array(fa.alibi_slopes(hq), dtype=np.float32)


@pytest.mark.parametrize("case", [
    PrefillCase("alibi_causal", B=2, Hq=8, Hkv=8, Nq=700, Nk=700, d=128, causal=True, seed=401),
    PrefillCase("alibi_noncausal", B=1, Hq=4, Hkv=2, Nq=300, Nk=500, d=64, seed=402),
    PrefillCase("alibi_window", B=1, Hq=8, Hkv=2, Nq=600, Nk=600, d=128, causal=True, window=200, seed=403),
    PrefillCase("alibi_gqa_q_lt_k", B=2, Hq=12, Hkv=4, Nq=130, Nk=900, d=128, causal=True, seed=404),
    PrefillCase("alibi_varlen", B=3, Hq=4, Hkv=4, Nq=500, Nk=500, d=64, layout="packed", causal=True,
                len_q=[500, 17, 256], seed=405),
], ids=lambda c: c.name)
def test_alibi_prefill_matches_oracle(case):
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(case)
    slopes = _slopes(case.Hq)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    if case.layout == "packed":
        cu = torch.tensor([0] + list(np.cumsum(x.len_q)), dtype=torch.int32, device="cuda")
        o, lse = fa.fa_fwd_varlen(q, k, v, cu, cu, max(x.len_q), max(x.len_k), causal=case.causal,
                                  window=case.window, scale=case.softmax_scale, alibi_slopes=slopes)
    else:
        o, lse = fa.fa_fwd(q, k, v, causal=case.causal, window=case.window, scale=case.softmax_scale,
                           alibi_slopes=slopes)
    torch.cuda.synchronize()
    rows = oracle.all_rows(x.len_q, case.Hq)
    go, gl = gather_prefill_rows(x, o, lse, rows)
    c = case
    ro, rl = oracle.attention_rows(bf16_bits(x.q.reshape(-1, c.Hq, c.d)), bf16_bits(x.k.reshape(-1, c.Hkv, c.d)),
                                   bf16_bits(x.v.reshape(-1, c.Hkv, c.d)), x.q_off, x.len_q, x.k_off, x.len_k,
                                   c.softmax_scale, c.causal, c.window, rows, alibi_slopes=slopes.astype(np.float64))
    check(go, gl, ro, rl, case.name)
    assert fa.fa_device_status() == 0


def test_alibi_llama7b_causal_full_size_every_row():
    # llama7b_causal with ALiBi, launched as the bench's ALiBi row launches it, every output row
    # against the oracle with the same slopes: the reverse walk, the chunk-bounded base of the
    # diagonal tile and the max-free later tiles across all 1,024 persistent items.  ALiBi makes
    # many rows follow one nearby key, so |O| reaches ~4.3 (a single V row), where bf16's half
    # spacing is 1.56e-2: no bf16 output meets the 1e-2 side of the rule there, and the derived
    # per-element bound (bf16 output and weight rounding) applies, as for other large-|O| cases.
    import flashattention_forward_fa_gb300 as fa
    from fa_workloads import LLAMA7B_CAUSAL
    from tests._util import prefill_parity_all_rows
    case = LLAMA7B_CAUSAL
    x = make_prefill(case)
    slopes = _slopes(case.Hq)
    o, lse = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True, scale=case.softmax_scale,
                       alibi_slopes=slopes)
    torch.cuda.synchronize()
    res = prefill_parity_all_rows(x, o, lse, case.name + "_alibi", strict=False,
                                  alibi_slopes=slopes.astype(np.float64))
    assert res["rows"] == case.B * case.Hq * case.Nq and res["empty_rows"] == 0
    assert res["o_bound_ratio"] <= 1.0
    assert fa.fa_device_status() == 0


def test_alibi_zero_slopes_equal_plain_prefill():
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(PrefillCase("z", B=1, Hq=4, Hkv=4, Nq=400, Nk=400, d=128, causal=True, seed=406))
    o1, l1 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True, alibi_slopes=np.zeros(4, np.float32))
    o2, l2 = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


@pytest.mark.parametrize("paged", [False, True])
def test_alibi_decode_matches_oracle(paged):
    import flashattention_forward_fa_gb300 as fa
    B, Hq, Hkv, d, page = 3, 16, 4, 128, 128
    lens = [1500, 129, 640]
    g = torch.Generator("cpu").manual_seed(407)
    cap = 1536
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, cap, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, cap, Hkv, d, generator=g).to(torch.bfloat16)
    slopes = _slopes(Hq)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    if paged:
        nb = cap // page
        table = torch.arange(B * nb, dtype=torch.int32).reshape(B, nb).flip(1).contiguous()  # reversed pages
        kp = torch.empty(B * nb, page, Hkv, d, dtype=torch.bfloat16)
        vp = torch.empty_like(kp)
        for b in range(B):
            for blk in range(nb):
                kp[table[b, blk]] = k[b, blk * page:(blk + 1) * page]
                vp[table[b, blk]] = v[b, blk * page:(blk + 1) * page]
        o, lse = fa.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens_dev, seqlens_k_host=lens,
                                    alibi_slopes=slopes)
    else:
        o, lse = fa.fa_decode(q.cuda(), k.cuda(), v.cuda(), lens_dev, seqlens_k_host=lens, alibi_slopes=slopes)
    torch.cuda.synchronize()
    rows = np.array([(b, h, 0) for b in range(B) for h in range(Hq)], dtype=np.int32)
    ro, rl = oracle.attention_rows(bf16_bits(q.reshape(B, 1, Hq, d)), bf16_bits(k), bf16_bits(v), list(range(B)),
                                   [1] * B, [b * cap for b in range(B)], lens, 1.0 / np.sqrt(d), True, 0, rows,
                                   alibi_slopes=slopes.astype(np.float64))
    go = o.float().cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    gl = lse.cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    check(go, gl, ro, rl, f"alibi decode paged={paged}")
    assert fa.fa_device_status() == 0
