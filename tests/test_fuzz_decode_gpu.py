"""Seeded random decode cases against the fp64 oracle: every (sequence, token, head) row.

Batch, head counts and grouping, head dim, cache capacity and per-sequence lengths (empty
ones included), new tokens per sequence, window, ALiBi, split count and a paged or
contiguous cache are drawn from one fixed generator, so that the split plan, the row blocks,
the chunk boundaries and the page lookups meet in combinations the named cases do not list.
The new tokens are the last Nq cache slots (token t at position len - Nq + t, bottom-right).
"""

import numpy as np
import pytest
import torch

import oracle
from fa_workloads import bf16_bits
from tests._util import abs_bits, check

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=4242):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        hkv = int(rng.choice([1, 2, 4, 8]))
        group = int(rng.choice([1, 2, 4, 8]))
        B = int(rng.integers(1, 7))
        nq = int(rng.choice([1, 1, 2, 4, 7]))
        paged = bool(rng.random() < 0.4)
        page = int(rng.choice([64, 128, 256])) if paged else 0
        ncap = int(rng.integers(64, 3000))
        if paged:
            ncap = ((ncap + page - 1) // page) * page
        lens = [int(rng.integers(0, ncap + 1)) for _ in range(B)]
        if rng.random() < 0.3:
            lens[int(rng.integers(0, B))] = 0
        window = int(rng.integers(1, 600)) if rng.random() < 0.3 else 0
        alibi = bool(rng.random() < 0.25)
        splits = int(rng.integers(1, 20)) if rng.random() < 0.4 else 0
        out.append(dict(name=f"r{i}_d{d}_h{hkv * group}x{hkv}_b{B}_nq{nq}" + (f"_page{page}" if paged else "") +
                        (f"_w{window}" if window else "") + ("_alibi" if alibi else "") +
                        (f"_s{splits}" if splits else ""),
                        d=d, Hq=hkv * group, Hkv=hkv, B=B, nq=nq, page=page, Ncap=ncap, lens=lens,
                        window=window, alibi=alibi, splits=splits, seed=7000 + i))
    return out


@pytest.mark.parametrize("c", _cases(), ids=lambda c: c["name"])
def test_random_decode_matches_oracle(c):
    import flashattention_forward_fa_gb300 as fa
    g = torch.Generator("cpu").manual_seed(c["seed"])
    B, nq, Hq, Hkv, d, ncap = c["B"], c["nq"], c["Hq"], c["Hkv"], c["d"], c["Ncap"]
    q = torch.randn(B, nq, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, ncap, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, ncap, Hkv, d, generator=g).to(torch.bfloat16)
    lens = c["lens"]
    scale = 1.0 / np.sqrt(d)
    slopes = np.array(fa.alibi_slopes(Hq), dtype=np.float32) if c["alibi"] else None
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qg = (q[:, 0] if nq == 1 else q).contiguous().cuda()
    if c["page"]:
        page = c["page"]
        nb = ncap // page
        perm = torch.randperm(B * nb, generator=g)
        kp = torch.empty((B * nb, page, Hkv, d), dtype=torch.bfloat16)
        vp = torch.empty_like(kp)
        kp[perm] = k.reshape(B * nb, page, Hkv, d)
        vp[perm] = v.reshape(B * nb, page, Hkv, d)
        table = perm.view(B, nb).to(torch.int32).contiguous().cuda()
        o, lse = fa.fa_decode_paged(qg, kp.cuda(), vp.cuda(), table, lens_dev, window=c["window"], scale=scale,
                                    num_splits=c["splits"], seqlens_k_host=lens, alibi_slopes=slopes)
    else:
        o, lse = fa.fa_decode(qg, k.cuda(), v.cuda(), lens_dev, window=c["window"], scale=scale,
                              num_splits=c["splits"], seqlens_k_host=lens, alibi_slopes=slopes)
    torch.cuda.synchronize()
    rows = oracle.all_rows([nq] * B, Hq)  # (b, h, t)
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    args = ([b * nq for b in range(B)], [nq] * B, [b * ncap for b in range(B)], lens, scale, True, c["window"], rows)
    sl = None if slopes is None else slopes.astype(np.float64)
    ro, rl = oracle.attention_rows(qb, kb, vb, *args, alibi_slopes=sl)
    oa, _ = oracle.attention_rows(qb, kb, abs_bits(vb), *args, alibi_slopes=sl)   # the same weights over |V|
    o4 = o.float().cpu().numpy().reshape(B, nq, Hq, d)
    l3 = lse.cpu().numpy().reshape(B, Hq, nq)
    go = o4[rows[:, 0], rows[:, 2], rows[:, 1]].astype(np.float64)
    gl = l3[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
    check(go, gl, ro, rl, c["name"], strict=False, o_abs=oa)
    assert torch.isfinite(o.float()).all()
    assert fa.fa_device_status() == 0
