"""GPU parity of the split-KV decode path (split kernel + combine) against the
fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from fa_workloads import DECODE_CACHE, DecodeCase, make_decode, shrink
from tests._util import check, gpu_decode, oracle_decode_rows

pytestmark = pytest.mark.gpu


def _all_pairs(B, Hq):
    return np.array([(b, h) for b in range(B) for h in range(Hq)], dtype=np.int32)


def _parity(case: DecodeCase, num_splits=0, with_host_lens=True, rows=None):
    import flashattention_forward_fa_gb300 as fa
    x = make_decode(case)
    o, lse = gpu_decode(x, num_splits=num_splits, with_host_lens=with_host_lens)
    rows = _all_pairs(case.B, case.Hq) if rows is None else rows
    go = o.float().cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    gl = lse.cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    ro, rl = oracle_decode_rows(x, rows)
    res = check(go, gl, ro, rl, case.name)
    assert fa.fa_device_status() == 0
    return x, o, lse, res


def test_decode_cache_full_size_every_row():
    # B=64, Hq=32, Hkv=8, d=128, cache 8192, lengths uniform in [512, 8192]: all 2048 (b, h) rows,
    # launched as the bench launches it (automatic split plan from the host lengths)
    x, o, lse, res = _parity(DECODE_CACHE)
    assert res["rows"] == 64 * 32 and res["empty_rows"] == 0 and res["o_loose_elems"] == 0


def test_decode_cache_reduced_full():
    _parity(shrink(DECODE_CACHE, name="decode_small", B=8, Ncap=2048, len_range=(1, 2048)))


@pytest.mark.parametrize("case", [
    DecodeCase("mha_d64", B=3, Hq=4, Hkv=4, Ncap=500, d=64, lens=[1, 63, 500], seed=41),
    DecodeCase("gqa8_d128", B=4, Hq=16, Hkv=2, Ncap=1000, d=128, lens=[64, 65, 999, 1000], seed=42),
    DecodeCase("mqa_g32", B=2, Hq=32, Hkv=1, Ncap=700, d=128, lens=[700, 129], seed=43),
    DecodeCase("g16_d64", B=2, Hq=16, Hkv=1, Ncap=300, d=64, lens=[257, 3], seed=44),
    DecodeCase("g3_odd", B=2, Hq=6, Hkv=2, Ncap=333, d=128, lens=[333, 200], seed=45),
    DecodeCase("empty_seq", B=3, Hq=8, Hkv=2, Ncap=256, d=128, lens=[0, 256, 1], seed=46),
    DecodeCase("window", B=3, Hq=8, Hkv=2, Ncap=1500, d=128, lens=[1500, 100, 700], window=256, seed=47),
    DecodeCase("window1", B=2, Hq=4, Hkv=1, Ncap=200, d=64, lens=[200, 5], window=1, seed=48),
], ids=lambda c: c.name)
def test_decode_edges(case):
    _parity(case)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 5, 8, 16, 33])
def test_every_split_count(num_splits):
    _parity(DecodeCase("splits", B=3, Hq=8, Hkv=2, Ncap=2100, d=128, lens=[2100, 1, 777], seed=49),
            num_splits=num_splits)


def test_split_count_invariance():
    # changing the split count only changes fp32 summation order
    case = DecodeCase("inv", B=4, Hq=8, Hkv=2, Ncap=4096, d=128, len_range=(1, 4096), seed=50)
    x = make_decode(case)
    outs = [gpu_decode(x, num_splits=s) for s in (1, 4, 16)]
    for o, l in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 1e-2
        assert (l - outs[0][1]).abs().max().item() <= 1e-3


def test_without_host_lengths_matches():
    case = DecodeCase("nohost", B=4, Hq=8, Hkv=2, Ncap=3000, d=128, len_range=(1, 3000), seed=51)
    _parity(case, with_host_lens=False)


def test_garbage_past_length_is_ignored():
    # cache slots past each sequence's length hold NaN/Inf: they must not leak into the output
    import flashattention_forward_fa_gb300 as fa
    case = DecodeCase("nan_tail", B=3, Hq=8, Hkv=2, Ncap=400, d=128, lens=[1, 130, 333], seed=52)
    x = make_decode(case)
    k = x.k_cache.clone()
    v = x.v_cache.clone()
    for b, n in enumerate(x.lens):
        k[b, n:] = float("nan")
        v[b, n:] = float("inf")
    lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
    o, lse = fa.fa_decode(x.q.cuda(), k.cuda(), v.cuda(), lens, seqlens_k_host=x.lens)
    torch.cuda.synchronize()
    ref_o, ref_l = gpu_decode(x)
    assert torch.isfinite(o.float()).all()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_decode_matches_prefill_last_row():
    # a decode step equals the last row of a causal prefill over the same keys
    import flashattention_forward_fa_gb300 as fa
    case = DecodeCase("vs_prefill", B=2, Hq=8, Hkv=2, Ncap=640, d=128, lens=[640, 640], seed=53)
    x = make_decode(case)
    o, lse = gpu_decode(x)
    q4 = x.q.reshape(2, 1, 8, 128).cuda()
    po, pl = fa.fa_fwd(q4, x.k_cache.cuda(), x.v_cache.cuda(), causal=True)
    assert (po[:, 0].float() - o.float()).abs().max().item() <= 1e-2
    assert (pl[:, :, 0] - lse).abs().max().item() <= 1e-3


def test_decode_replays_from_cuda_graph():
    # a serving loop captures the decode once and replays it per token with new inputs in the same
    # buffers: the captured launches must read the buffers at replay time and match eager calls
    import flashattention_forward_fa_gb300 as fa
    c = shrink(DECODE_CACHE, name="graph", B=8, Ncap=2048, len_range=(100, 2048), seed=71)
    x = make_decode(c)
    q, kc, vc = x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda()
    lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
    S = fa.fa_decode_max_splits(c.B, c.Hq, c.Hkv, c.Ncap, 0, x.lens, 0)
    ws = torch.empty((fa.decode_workspace_size(c.B, c.Hq, c.d, S) + 3) // 4, dtype=torch.float32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((c.B, c.Hq), dtype=torch.float32, device="cuda")
    fa.fa_decode(q, kc, vc, lens, seqlens_k_host=x.lens, workspace=ws, out=o, lse=lse)  # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.fa_decode(q, kc, vc, lens, seqlens_k_host=x.lens, workspace=ws, out=o, lse=lse)
    gen = torch.Generator("cpu").manual_seed(72)
    for step in range(3):
        q.copy_(torch.randn(q.shape, generator=gen).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        o_ref, lse_ref = fa.fa_decode(q, kc, vc, lens, seqlens_k_host=x.lens)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), f"replay {step} differs from an eager call"
    assert fa.fa_device_status() == 0


def test_understated_host_lengths_are_reported():
    # the host copy of the lengths plans the splits; one that understates the device lengths leaves
    # keys unread, which the combine kernel reports as a bounds error (bit 1) instead of silently
    import flashattention_forward_fa_gb300 as fa
    case = DecodeCase("understated", B=3, Hq=8, Hkv=2, Ncap=2048, d=128, lens=[2048, 1000, 64], seed=54)
    x = make_decode(case)
    lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
    fa.fa_device_status(clear=True)
    o, lse = fa.fa_decode(x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), lens, num_splits=2,
                          seqlens_k_host=[n // 4 for n in x.lens])
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) & 2
    assert torch.isfinite(o.float()).all()
    # an overstated host copy is fine: the same outputs as with the exact one, no error bit
    o1, l1 = fa.fa_decode(x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), lens, num_splits=2,
                          seqlens_k_host=x.lens)
    o2, l2 = fa.fa_decode(x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), lens, num_splits=2,
                          seqlens_k_host=[case.Ncap] * case.B)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == 0
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2 and (l1 - l2).abs().max().item() <= 1e-3
