"""Seeded random prefill cases against the fp64 oracle: every output row of each case.

The named workloads and the edge grid pin chosen shapes; these cases draw head counts,
grouping, head dim, lengths, layout, causal/window masks and ALiBi at random (fixed seed), so
that items of every kind meet in one launch: head pairs and row-tile pairs, persistent and
one-CTA-per-item grids, tiles that are staged for TMA stores next to ragged ones, several
items per CTA, sequences without rows or without keys.
"""

import numpy as np
import pytest
import torch

from fa_workloads import PrefillCase, make_prefill
from tests._util import prefill_parity_all_rows

pytestmark = pytest.mark.gpu


def _cases(n=32, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        hkv = int(rng.choice([1, 2, 4]))
        group = int(rng.choice([1, 2, 3, 4, 8]))
        hq = hkv * group
        B = int(rng.integers(1, 5))
        layout = str(rng.choice(["dense", "padded", "packed"]))
        causal = bool(rng.random() < 0.6)
        window = int(rng.integers(1, 400)) if rng.random() < 0.35 else 0
        alibi = bool(rng.random() < 0.25)
        k_mult = float(rng.choice([1.0, 1.0, 3.0]))
        nq = int(rng.integers(1, 700))
        nk = nq if (causal and rng.random() < 0.5) else int(rng.integers(1, 800))
        len_q = len_k = None
        if layout == "padded":
            len_q = [int(rng.integers(0, nq + 1)) for _ in range(B)]
            len_k = [int(rng.integers(0, nk + 1)) for _ in range(B)]
        elif layout == "packed":
            len_q = [int(rng.integers(0, 600)) for _ in range(B)]
            len_k = [int(rng.integers(0, 700)) for _ in range(B)]
            len_q[0] = max(len_q[0], 1)
            len_k[0] = max(len_k[0], 1)  # keep the packed K/V tensors non-empty
            nq, nk = max(len_q), max(len_k)
        name = (f"r{i}_{layout}_d{d}_h{hq}x{hkv}_b{B}" + ("_causal" if causal else "") +
                (f"_w{window}" if window else "") + ("_alibi" if alibi else ""))
        case = PrefillCase(name, B=B, Hq=hq, Hkv=hkv, Nq=nq, Nk=nk, d=d, causal=causal, window=window,
                           layout=layout, len_q=len_q, len_k=len_k, k_mult=k_mult, seed=5000 + i)
        out.append((case, alibi))
    return out


@pytest.mark.parametrize("case,alibi", _cases(), ids=lambda c: c.name if isinstance(c, PrefillCase) else str(c))
def test_random_prefill_matches_oracle(case, alibi):
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(case)
    slopes = np.array(fa.alibi_slopes(case.Hq), dtype=np.float32) if alibi else None
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    if case.layout == "packed":
        cu_q = torch.tensor([0] + list(np.cumsum(x.len_q)), dtype=torch.int32, device="cuda")
        cu_k = torch.tensor([0] + list(np.cumsum(x.len_k)), dtype=torch.int32, device="cuda")
        o, lse = fa.fa_fwd_varlen(q, k, v, cu_q, cu_k, max(x.len_q), max(x.len_k), causal=case.causal,
                                  window=case.window, scale=case.softmax_scale, alibi_slopes=slopes)
    elif case.layout == "padded":
        sq = torch.tensor(x.len_q, dtype=torch.int32, device="cuda")
        sk = torch.tensor(x.len_k, dtype=torch.int32, device="cuda")
        o, lse = fa.fa_fwd(q, k, v, causal=case.causal, window=case.window, scale=case.softmax_scale,
                           seqlens_q=sq, seqlens_k=sk, alibi_slopes=slopes)
    else:
        o, lse = fa.fa_fwd(q, k, v, causal=case.causal, window=case.window, scale=case.softmax_scale,
                           alibi_slopes=slopes)
    torch.cuda.synchronize()
    # rows that see few keys (short sequences, narrow windows, sharpened scores) can reach |O| > 1.28,
    # where bf16 output rounding alone exceeds 1e-2: the derived per-element bound applies
    prefill_parity_all_rows(x, o, lse, case.name, strict=False, alibi_slopes=slopes)
    if case.layout == "padded":
        for b, lq in enumerate(x.len_q):
            assert torch.all(o[b, lq:] == 0)
    assert torch.isfinite(o.float()).all()
    assert fa.fa_device_status() == 0
