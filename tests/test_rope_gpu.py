"""RoPE (jsqmd page, §三 "RoPE的设计动机与计算特点" and "融合位置编码的Attention计算"):
the rotation kernel against the oracle's rotation, and the prefill with Q rotated inside
the kernel (K rotated once beforehand) against the oracle's attention over the oracle's
rotated Q and K."""

import numpy as np
import pytest
import torch

import oracle
from oracle import rope as orope
from fa_workloads import PrefillCase, bf16_bits, make_prefill
from tests._util import check, gather_prefill_rows

pytestmark = pytest.mark.gpu


def _tables(max_pos, rd):
    import flashattention_forward_fa_gb300 as fa
    return fa.rope_tables(max_pos, rd, device="cuda")


def _bf16_pattern_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# The first four shapes run the one-thread-per-chunk form of the kernel, the last three (rows of
# at least 512 16-byte chunks) the one-row-per-CTA form, including 15 chunks per head (threads
# past the last whole group idle) and a row that takes one pass of four heads per thread.
@pytest.mark.parametrize("rows,H,d,rd", [(1000, 8, 128, 128), (333, 2, 64, 64), (77, 4, 128, 64), (5, 1, 64, 8),
                                         (300, 32, 128, 128), (129, 40, 128, 120), (64, 64, 64, 64)])
def test_rope_kernel_matches_oracle(rows, H, d, rd):
    # Tolerance derived from the kernel's arithmetic.  The kernel rotates a pair (x, y) in fp32 as
    # fma(x, c, -(y s)) and fma(x, s, y c) with the fp32 table values c, s, then rounds to bf16
    # (nearest even).  Each fp32 result r32 is within 2^-24 |y s| + 2^-24 |r| <= 2^-23 (|x| + |y|)
    # of the exact rotation r with the same tables (|c|, |s| <= 1), so the kernel's bf16 value g is
    # the rounding of some value within delta = 2^-22 (|x| + |y|) of r (a factor 2 of margin):
    # |g - r| <= h(g) + delta, h(g) the larger half-spacing of bf16 values next to g.  Where no
    # rounding boundary lies within delta of r, that forces g to equal the oracle's single RNE
    # rounding of r; elsewhere (near boundaries, or when cancellation makes r tiny next to delta)
    # g may differ from it by what delta allows.
    import flashattention_forward_fa_gb300 as fa
    g = torch.Generator("cpu").manual_seed(rows + rd)
    x = torch.randn(rows, H, d, generator=g).to(torch.bfloat16)
    pos = torch.randint(0, 4096, (rows,), generator=g, dtype=torch.int32)
    cos_t, sin_t = _tables(4096, rd)
    y = fa.fa_rope(x.cuda(), pos.cuda(), (cos_t, sin_t))
    torch.cuda.synchronize()
    x64 = x.to(torch.float64).numpy()
    exact = orope.rotate(x64, pos.numpy(), cos_t.cpu().double().numpy(), sin_t.cpu().double().numpy(), rd)
    ref_bits = orope.bf16_round_bits(exact)
    got_bits = y.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_bits[..., rd:], x.view(torch.int16).numpy().view(np.uint16)[..., rd:])
    pair = np.abs(x64[..., :rd:2]) + np.abs(x64[..., 1:rd:2])          # |x| + |y| of each element's pair
    delta = np.ldexp(np.repeat(pair, 2, axis=-1), -22)
    gv = _bf16_pattern_value(got_bits[..., :rd])
    _, e = np.frexp(np.abs(gv))
    h = np.ldexp(1.0, np.maximum(e, -125) - 9)                         # half the spacing above |g|
    dist = np.abs(gv - exact[..., :rd])
    assert np.all(dist <= h + delta), f"worst |g - r| / (h + delta) = {float((dist / (h + delta)).max()):.2f}"
    # and where no rounding boundary is within delta of r, g is the oracle's value bit for bit
    rv = _bf16_pattern_value(ref_bits[..., :rd])
    mr, er = np.frexp(np.abs(rv))
    # half the spacing next to ref; a power of two has the finer spacing of the binade below it
    hr = np.ldexp(1.0, np.maximum(er, -125) - np.where(mr == 0.5, 10, 9))
    clear = np.abs(exact[..., :rd] - rv) + delta < hr
    assert np.array_equal(got_bits[..., :rd][clear], ref_bits[..., :rd][clear])
    assert clear.mean() > 0.95
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("H,d", [(2, 64), (32, 128)])
def test_rope_position_out_of_table_reported(H, d):
    import flashattention_forward_fa_gb300 as fa
    x = torch.randn(4, H, d).to(torch.bfloat16).cuda()
    x0 = x.clone()
    pos = torch.tensor([0, 1, 99, 2], dtype=torch.int32, device="cuda")
    fa.fa_device_status(clear=True)
    fa.fa_rope(x, pos, _tables(16, d))
    assert fa.fa_device_status(clear=True) & 2
    assert torch.equal(x[2], x0[2])
    assert not torch.equal(x[3], x0[3])  # the rows around it are still rotated


def _oracle_rope_prefill(x, case, cos64, sin64, rd):
    c = case
    qs, ks = [], []
    q3 = x.q.reshape(-1, c.Hq, c.d)
    k3 = x.k.reshape(-1, c.Hkv, c.d)
    q_pos = np.zeros(q3.shape[0], np.int64)
    k_pos = np.zeros(k3.shape[0], np.int64)
    for b in range(len(x.len_q)):
        lq, lk = x.len_q[b], x.len_k[b]
        q_pos[x.q_off[b]:x.q_off[b] + lq] = np.arange(lq) + lk - lq    # bottom-right positions
        k_pos[x.k_off[b]:x.k_off[b] + lk] = np.arange(lk)
    qr = orope.rotate_bf16(q3, q_pos, cos64, sin64, rd)
    kr = orope.rotate_bf16(k3, k_pos, cos64, sin64, rd)
    rows = oracle.all_rows(x.len_q, c.Hq)
    ro, rl = oracle.attention_rows(bf16_bits(qr), bf16_bits(kr), bf16_bits(x.v.reshape(-1, c.Hkv, c.d)), x.q_off,
                                   x.len_q, x.k_off, x.len_k, c.softmax_scale, c.causal, c.window, rows)
    return rows, ro, rl, k_pos


@pytest.mark.parametrize("case,rd", [
    (PrefillCase("rope_causal", B=2, Hq=8, Hkv=8, Nq=700, Nk=700, d=128, causal=True, seed=501), 128),
    (PrefillCase("rope_gqa_q_lt_k", B=2, Hq=12, Hkv=4, Nq=130, Nk=900, d=128, causal=True, seed=502), 128),
    (PrefillCase("rope_partial_d64", B=1, Hq=4, Hkv=2, Nq=300, Nk=500, d=64, seed=503), 32),
    (PrefillCase("rope_window", B=1, Hq=8, Hkv=2, Nq=600, Nk=600, d=128, causal=True, window=200, seed=504), 64),
    (PrefillCase("rope_varlen", B=3, Hq=4, Hkv=4, Nq=500, Nk=500, d=64, layout="packed", causal=True,
                 len_q=[500, 17, 256], seed=505), 64),
    (PrefillCase("rope_dim40_tail", B=1, Hq=4, Hkv=4, Nq=384, Nk=384, d=128, causal=True, seed=508), 40),
], ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_fused_rope_prefill_matches_oracle(case, rd):
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(case)
    cos_t, sin_t = _tables(1024, rd)
    cos64, sin64 = cos_t.cpu().double().numpy(), sin_t.cpu().double().numpy()
    rows, ro, rl, k_pos = _oracle_rope_prefill(x, case, cos64, sin64, rd)
    q, v = x.q.cuda(), x.v.cuda()
    k = x.k.cuda().clone()
    fa.fa_rope(k, torch.from_numpy(k_pos).to(torch.int32).cuda(), (cos_t, sin_t))   # K rotated once
    if case.layout == "packed":
        cu = torch.tensor([0] + list(np.cumsum(x.len_q)), dtype=torch.int32, device="cuda")
        o, lse = fa.fa_fwd_varlen(q, k, v, cu, cu, max(x.len_q), max(x.len_k), causal=case.causal,
                                  window=case.window, scale=case.softmax_scale, rope=(cos_t, sin_t))
    else:
        o, lse = fa.fa_fwd(q, k, v, causal=case.causal, window=case.window, scale=case.softmax_scale,
                           rope=(cos_t, sin_t))
    torch.cuda.synchronize()
    go, gl = gather_prefill_rows(x, o, lse, rows)
    check(go, gl, ro, rl, case.name)
    assert fa.fa_device_status() == 0


def test_fused_rope_with_alibi():
    # both position schemes at once exercise the <ALIBI, ROPE> kernel variant
    import flashattention_forward_fa_gb300 as fa
    case = PrefillCase("rope_alibi", B=1, Hq=4, Hkv=4, Nq=400, Nk=400, d=128, causal=True, seed=506)
    x = make_prefill(case)
    cos_t, sin_t = _tables(512, 128)
    cos64, sin64 = cos_t.cpu().double().numpy(), sin_t.cpu().double().numpy()
    slopes = np.array(fa.alibi_slopes(4), np.float32)
    q3, k3 = x.q.reshape(-1, 4, 128), x.k.reshape(-1, 4, 128)
    qr = orope.rotate_bf16(q3, np.arange(400), cos64, sin64, 128)
    kr = orope.rotate_bf16(k3, np.arange(400), cos64, sin64, 128)
    rows = oracle.all_rows(x.len_q, 4)
    ro, rl = oracle.attention_rows(bf16_bits(qr), bf16_bits(kr), bf16_bits(x.v.reshape(-1, 4, 128)), x.q_off,
                                   x.len_q, x.k_off, x.len_k, case.softmax_scale, True, 0, rows,
                                   alibi_slopes=slopes.astype(np.float64))
    k = x.k.cuda().clone()
    fa.fa_rope(k, torch.arange(400, dtype=torch.int32, device="cuda"), (cos_t, sin_t))
    o, lse = fa.fa_fwd(x.q.cuda(), k, x.v.cuda(), causal=True, alibi_slopes=slopes, rope=(cos_t, sin_t))
    torch.cuda.synchronize()
    go, gl = gather_prefill_rows(x, o, lse, rows)
    check(go, gl, ro, rl, case.name)
    assert fa.fa_device_status() == 0


def test_query_position_past_table_reported():
    import flashattention_forward_fa_gb300 as fa
    x = make_prefill(PrefillCase("short_table", B=1, Hq=2, Hkv=2, Nq=200, Nk=200, d=64, seed=507))
    cos_t, sin_t = _tables(100, 64)       # positions 100..199 have no table row
    fa.fa_device_status(clear=True)
    o, lse = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), rope=(cos_t, sin_t))
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) & 2
    assert torch.isfinite(o.float()).all()
