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
    # Tolerance derived from the kernel's arithmetic.  The kernel rotates a pair (x, y) in fp32
    # with the fp32 table values c, s: it splits y s into its rounding p and the exact error
    # e = fma(y, s, -p) and computes fma(x, c, -p) - e (likewise x s + y c), then rounds to bf16
    # (nearest even).  With t = fma(x, c, -p) = (x c - p)(1 + d1) and the subtraction rounded by
    # (1 + d2), |d1|, |d2| <= 2^-24, the fp32 result is within 2^-23 |r| + 2^-48 |y| (to first
    # order) of the exact rotation r with the same tables, so the kernel's bf16 value g is the
    # rounding of some value within delta = 2^-22 |r| + 2^-46 (|x| + |y|) of r (a factor 2 and 4
    # of margin): |g - r| <= h(g) + delta, h(g) the larger half-spacing of bf16 values next to g.
    # Where no rounding boundary lies within delta of r, that forces g to equal the oracle's
    # single RNE rounding of r, which is then required bit for bit (all but a few elements).
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
    delta = np.ldexp(np.abs(exact[..., :rd]), -22) + np.ldexp(np.repeat(pair, 2, axis=-1), -46)
    gv = _bf16_pattern_value(got_bits[..., :rd])
    _, e = np.frexp(np.abs(gv))
    h = np.ldexp(1.0, np.maximum(e, -125) - 9)                         # half the spacing above |g|
    dist = np.abs(gv - exact[..., :rd])
    assert np.all(dist <= h + delta), f"worst |g - r| / (h + delta) = {float((dist / (h + delta)).max()):.2f}"
    # and where no rounding boundary is within delta of r, g is the oracle's value bit for bit
    rv = _bf16_pattern_value(ref_bits[..., :rd])
    mr, er = np.frexp(np.abs(rv))
    # half the spacing on r's side of ref: below a power of two the binade below's finer spacing
    above = np.abs(exact[..., :rd]) >= np.abs(rv)
    hr = np.ldexp(1.0, np.maximum(er, -125) - np.where((mr == 0.5) & ~above, 10, 9))
    clear = np.abs(exact[..., :rd] - rv) + delta < hr
    assert np.array_equal(got_bits[..., :rd][clear], ref_bits[..., :rd][clear])
    assert clear.mean() > 0.999
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


def _near_boundary(x_bf16: torch.Tensor, exact: np.ndarray, rd: int, widen: float = 1.0):
    """Elements of a rotation whose exact value lies so close to a bf16 rounding boundary that the
    kernel's fp32 arithmetic (within 2^-22 |r| + 2^-46 (|x| + |y|) of it, see the tolerance above)
    may round it to the other neighbour: a mask over the rotated dimensions and the bf16 spacing
    there (the size of such a flip).  ``widen`` scales the margin (the CPU check of the allowance
    uses a wide one so that a small problem has many such elements)."""
    x64 = x_bf16.to(torch.float64).numpy()
    ex = exact[..., :rd]
    rv = (orope.bf16_round_bits(exact)[..., :rd].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    mr, er = np.frexp(np.abs(rv))
    above = np.abs(ex) >= np.abs(rv)
    hr = np.ldexp(1.0, np.maximum(er, -125) - np.where((mr == 0.5) & ~above, 10, 9))
    pair = np.abs(x64[..., :rd:2]) + np.abs(x64[..., 1:rd:2])
    delta = widen * (np.ldexp(np.abs(ex), -22) + np.ldexp(np.repeat(pair, 2, axis=-1), -46))
    near = np.abs(ex - rv) + delta >= hr
    return near, 2.0 * np.ldexp(1.0, np.maximum(er, -125) - 9)   # a flip moves by at most one spacing


def _rope_flip_allowance(x, qr, kr, q_ex, k_ex, rd, scale, lse_ref, widen: float = 1.0, max_frac: float = 1e-4):
    """[N, H] bound on how far the LSE of causal row i of head h (one sequence, Hq = Hkv) may move
    when boundary elements of the rotated Q and K round to their other neighbour.  Row i's scores
    change by ds_j = x_j + y_j: x_j = scale dq . k_j from its own flips dq, y_j from key j's flips
    (|y_j| <= b_j = scale x key j's flip sizes x this row's |q| there, zero for keys without flips).
    By Jensen and Hoeffding's lemma, |dLSE| = |log sum_j p_j e^(ds_j)| <= |E_p ds| + r^2 / 2 with
    |ds_j| <= r, and |E_p ds| <= scale sum_d |dq_d| |E_p k_d| + sum_j p_j b_j, p the oracle's
    attention weights (E_p k is the oracle's attention of the row over K as values)."""
    c = x.case
    q3, k3 = x.q.reshape(-1, c.Hq, c.d), x.k.reshape(-1, c.Hkv, c.d)
    nq, sq = _near_boundary(q3, q_ex, rd, widen)
    nk, sk = _near_boundary(k3, k_ex, rd, widen)
    assert nq.mean() < max_frac and nk.mean() < max_frac
    qv = qr.to(torch.float64).numpy()
    kv = kr.to(torch.float64).numpy()
    qa = np.abs(qv[..., :rd]) + sq   # |q| after a possible flip
    ka = np.abs(kv[..., :rd]) + sk
    n, heads = qv.shape[0], qv.shape[1]
    rows = np.arange(n)
    # own flips: |E_p x| <= scale sum_d dq_d |E_p k_d|, for the rows that have any
    xterm, xmax = np.zeros((n, heads)), scale * (nq * sq * ka.max(axis=0)[None]).sum(-1)
    ii, hh = np.nonzero(nq.any(-1))
    if len(ii):
        trip = np.stack([np.zeros_like(ii), hh, ii], 1).astype(np.int32)
        ek, _ = oracle.attention_rows(bf16_bits(qr), bf16_bits(kr), bf16_bits(kr), x.q_off, x.len_q, x.k_off,
                                      x.len_k, scale, True, 0, trip)
        xterm[ii, hh] = scale * (nq[ii, hh] * sq[ii, hh] * np.abs(ek[:, :rd])).sum(-1)
    # key flips: sum_j p_j b_j and max_j b_j over the visible keys with flips
    yterm, ymax = np.zeros((n, heads)), np.zeros((n, heads))
    for h in range(heads):
        keys = np.unique(np.nonzero(nk[:, h, :])[0])
        if not len(keys):
            continue
        vis = rows[:, None] >= keys[None, :]                        # causal: key j visible from rows >= j
        p_f = np.exp(scale * (qv[:, h, :] @ kv[keys, h, :].T) - lse_ref[:, h][:, None]) * vis
        b = scale * (qa[:, h, :] @ (nk[keys, h, :] * sk[keys, h, :]).T) * vis
        yterm[:, h] = (p_f * b).sum(-1)
        ymax[:, h] = b.max(-1)
    r = xmax + ymax
    return xterm + yterm + r * r / 2.0 + 1e-6                      # + rounding of the bound itself


def test_fused_rope_llama7b_causal_full_size_every_row():
    # llama7b_causal with Q rotated inside the kernel, set up as the bench's RoPE row (tables of
    # 8192 positions, rotary_dim 128, K rotated once by fa_rope at positions 0..N-1): every output
    # row against the oracle run on the single-rounded fp64 rotations of Q and K.  O is held to the
    # acceptance numbers.  The LSE is held to 1e-3 plus what the rotation's rounding may move it
    # by: a few elements of Q and K (~1e-5 of them) lie within the kernel's fp32 error of a bf16
    # rounding boundary, where either neighbour is a faithful rotation, and a flipped element moves
    # a score by at most scale x spacing x the largest |value| it multiplies; the LSE moves by at
    # most the largest score change of the row (its own query flips plus those of any visible key).
    import flashattention_forward_fa_gb300 as fa
    from fa_workloads import LLAMA7B_CAUSAL
    from tests._util import LSE_MAX_ABS, O_MAX_ABS, O_REL_RMS, PrefillOracle, host_outputs
    import dataclasses
    case = LLAMA7B_CAUSAL
    x = make_prefill(case)
    rd, H, N = case.d, case.Hq, case.Nq
    cos_t, sin_t = _tables(case.Nk, rd)
    cos64, sin64 = cos_t.cpu().double().numpy(), sin_t.cpu().double().numpy()
    pos = np.arange(case.Nk)  # one sequence, Nq = Nk: query and key positions coincide
    q3, k3 = x.q.reshape(-1, H, case.d), x.k.reshape(-1, case.Hkv, case.d)
    q_ex = orope.rotate(q3.to(torch.float64).numpy(), pos, cos64, sin64, rd)
    k_ex = orope.rotate(k3.to(torch.float64).numpy(), pos, cos64, sin64, rd)
    qr = orope.rotate_bf16(q3, pos, cos64, sin64, rd)
    kr = orope.rotate_bf16(k3, pos, cos64, sin64, rd)
    k = x.k.cuda().clone()
    fa.fa_rope(k, torch.from_numpy(pos).to(torch.int32).cuda(), (cos_t, sin_t))
    o, lse = fa.fa_fwd(x.q.cuda(), k, x.v.cuda(), causal=True, scale=case.softmax_scale, rope=(cos_t, sin_t))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    orc = PrefillOracle(dataclasses.replace(x, q=qr.reshape(x.q.shape), k=kr.reshape(x.k.shape)))
    oh, lh = host_outputs(o, lse)
    rows = oracle.all_rows(x.len_q, H)
    lse_ref, lse_gpu = np.zeros((N, H)), np.zeros((N, H))
    max_o, sq_err, sq_ref = 0.0, 0.0, 0.0
    for s0 in range(0, len(rows), 1 << 16):
        r = rows[s0:s0 + (1 << 16)]
        go, gl = gather_prefill_rows(x, oh, lh, r)
        ro, rl = orc.rows(r)
        assert np.all(np.isfinite(rl)) and np.all(np.isfinite(go))
        d = np.abs(go - ro)
        max_o = max(max_o, float(d.max()))
        sq_err += float((d ** 2).sum())
        sq_ref += float((ro ** 2).sum())
        lse_ref[r[:, 2], r[:, 1]] = rl
        lse_gpu[r[:, 2], r[:, 1]] = gl
    assert max_o <= O_MAX_ABS, f"O max-abs {max_o:.3e}"
    assert (sq_err / sq_ref) ** 0.5 <= O_REL_RMS
    # per-row LSE allowance: the acceptance number plus what boundary flips may add (Hq = Hkv)
    allow = LSE_MAX_ABS + _rope_flip_allowance(x, qr, kr, q_ex, k_ex, rd, case.softmax_scale, lse_ref)
    ratio = np.abs(lse_gpu - lse_ref) / allow
    assert ratio.max() <= 1.0, f"LSE error {ratio.max():.3f} x its allowance"


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
