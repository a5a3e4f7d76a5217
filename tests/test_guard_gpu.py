"""Out-of-bounds writes: every output buffer of a call sits inside a larger allocation whose
margins before and after are filled with a sentinel bit pattern; after the call the margins
must be bit-identical, and the outputs themselves must match the oracle.

A tail tile that writes past its sequence or past the end of the tensor (the failure the
agent.csdn.net BERT walkthrough, 第四章, runs into as a core dump) would change a margin.
The cases put ragged tiles everywhere: sequences of 1, 63, 65, 129 and 1000 rows, with the
last one ending exactly at the end of the packed tensor, padded batches with short valid
lengths, dense tensors whose last tile is partial, head-pair items, and the decode outputs,
split workspace and the in-place rotation.
"""

import numpy as np
import pytest
import torch

from fa_workloads import DecodeCase, PrefillCase, make_decode, make_prefill
from tests._util import check, oracle_decode_rows, prefill_parity_all_rows

pytestmark = pytest.mark.gpu

SENT16 = 0x7FA5           # a bf16 NaN pattern
SENT32 = 0x7FC0A5A5       # an fp32 NaN pattern


class Guarded:
    """An output tensor of ``shape`` placed ``margin`` elements into a sentinel-filled buffer."""

    def __init__(self, shape, dtype, margin):
        n = int(np.prod(shape))
        assert margin % 8 == 0                                   # keeps the view 16-byte aligned
        self.n, self.margin = n, margin
        if dtype == torch.bfloat16:
            self.buf = torch.full((margin + n + margin,), SENT16, dtype=torch.int16, device="cuda")
            self.sent = SENT16
        else:
            self.buf = torch.full((margin + n + margin,), SENT32, dtype=torch.int32, device="cuda")
            self.sent = SENT32
        self.t = self.buf[margin:margin + n].view(dtype).view(shape)
        assert self.t.data_ptr() % 16 == 0

    def assert_margins_intact(self, what):
        torch.cuda.synchronize()
        head, tail = self.buf[:self.margin], self.buf[self.margin + self.n:]
        bad_h = int((head != self.sent).sum())
        bad_t = int((tail != self.sent).sum())
        assert bad_h == 0 and bad_t == 0, f"{what}: {bad_h} elements before and {bad_t} after the output changed"


LENS = [1, 63, 65, 129, 1000]


def _prefill_outputs(x):
    c = x.case
    if c.layout == "packed":
        oshape, lshape = (sum(x.len_q), c.Hq, c.d), (c.Hq, sum(x.len_q))
    else:
        oshape, lshape = (c.B, c.Nq, c.Hq, c.d), (c.B, c.Hq, c.Nq)
    margin_o = 129 * c.Hq * c.d                                  # more than one 128-row tile
    return Guarded(oshape, torch.bfloat16, margin_o), Guarded(lshape, torch.float32, 1024)


PREFILL_CASES = [
    PrefillCase("packed_causal_d128", B=5, Hq=4, Hkv=2, Nq=1000, Nk=1000, d=128, layout="packed", causal=True,
                len_q=LENS, seed=901),
    PrefillCase("packed_noncausal_d64", B=5, Hq=2, Hkv=1, Nq=1000, Nk=1000, d=64, layout="packed",
                len_q=LENS, len_k=[7, 300, 1, 129, 1000], seed=902),
    PrefillCase("packed_window_gqa4", B=5, Hq=8, Hkv=2, Nq=1000, Nk=1000, d=128, layout="packed", causal=True,
                window=100, len_q=LENS, seed=903),
    PrefillCase("padded_seqlens_d128", B=5, Hq=2, Hkv=2, Nq=1000, Nk=1000, d=128, layout="padded", causal=True,
                len_q=[1000, 63, 65, 129, 1], len_k=[1000, 63, 70, 129, 1], seed=904),
    PrefillCase("dense_ragged_d64", B=2, Hq=2, Hkv=2, Nq=1000, Nk=1000, d=64, causal=True, seed=905),
    PrefillCase("dense_pair_heads_65", B=1, Hq=4, Hkv=2, Nq=65, Nk=65, d=128, causal=True, seed=906),
    PrefillCase("dense_63_noncausal", B=3, Hq=2, Hkv=1, Nq=63, Nk=129, d=128, seed=907),
    PrefillCase("dense_one_row", B=1, Hq=2, Hkv=2, Nq=1, Nk=1, d=64, seed=908),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: c.name)
def test_prefill_writes_stay_inside_outputs(case):
    import flashattention_forward_fa_gb300 as fa
    from tests._util import gpu_prefill
    x = make_prefill(case)
    go, gl = _prefill_outputs(x)
    o, lse = gpu_prefill(x, out=go.t, lse=gl.t)
    assert o.data_ptr() == go.t.data_ptr() and lse.data_ptr() == gl.t.data_ptr()
    go.assert_margins_intact(f"{case.name} O")
    gl.assert_margins_intact(f"{case.name} LSE")
    prefill_parity_all_rows(x, o, lse, case.name)
    if case.layout == "padded":
        for b, lq in enumerate(x.len_q):
            assert torch.all(o[b, lq:] == 0) and torch.all(torch.isneginf(lse[b, :, lq:]))
    assert fa.fa_device_status() == 0


def test_prefill_alibi_and_rope_writes_stay_inside_outputs():
    import flashattention_forward_fa_gb300 as fa
    case = PrefillCase("packed_alibi_rope", B=5, Hq=4, Hkv=4, Nq=1000, Nk=1000, d=128, layout="packed",
                       causal=True, len_q=LENS, seed=909)
    x = make_prefill(case)
    cu = torch.tensor([0] + list(np.cumsum(x.len_q)), dtype=torch.int32, device="cuda")
    slopes = torch.tensor(fa.alibi_slopes(case.Hq), dtype=torch.float32, device="cuda")
    cos_t, sin_t = fa.rope_tables(1024, 128, device="cuda")
    for kw in ({"alibi_slopes": slopes}, {"rope": (cos_t, sin_t)}):
        go, gl = _prefill_outputs(x)
        fa.fa_fwd_varlen(x.q.cuda(), x.k.cuda(), x.v.cuda(), cu, cu, 1000, 1000, causal=True, out=go.t, lse=gl.t,
                         **kw)
        go.assert_margins_intact(f"{case.name} {list(kw)} O")
        gl.assert_margins_intact(f"{case.name} {list(kw)} LSE")
        assert torch.isfinite(go.t.float()).all() and not torch.isnan(gl.t).any()
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("nq,paged", [(1, False), (3, False), (1, True), (2, True)],
                         ids=["one_token", "three_tokens", "paged", "paged_two_tokens"])
def test_decode_writes_stay_inside_outputs_and_workspace(nq, paged):
    import flashattention_forward_fa_gb300 as fa
    case = DecodeCase("guard_decode", B=5, Hq=8, Hkv=2, Ncap=1024, d=128, lens=[1, 63, 65, 129, 1024], seed=910)
    x = make_decode(case)
    g = torch.Generator("cpu").manual_seed(911)
    q = x.q if nq == 1 else torch.randn(case.B, nq, case.Hq, case.d, generator=g).to(torch.bfloat16)
    lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
    oshape = (case.B, case.Hq, case.d) if nq == 1 else (case.B, nq, case.Hq, case.d)
    lshape = (case.B, case.Hq) if nq == 1 else (case.B, case.Hq, nq)
    go = Guarded(oshape, torch.bfloat16, 1024)
    gl = Guarded(lshape, torch.float32, 1024)
    splits = 5
    ws_elems = (fa.decode_workspace_size(case.B * nq, case.Hq, case.d, splits) + 3) // 4
    gw = Guarded((ws_elems,), torch.float32, 1024)
    if paged:
        page = 128
        nb = case.Ncap // page
        perm = torch.randperm(case.B * nb, generator=g)
        kp = torch.empty((case.B * nb, page, case.Hkv, case.d), dtype=torch.bfloat16)
        vp = torch.empty_like(kp)
        kp[perm] = x.k_cache.reshape(case.B * nb, page, case.Hkv, case.d)
        vp[perm] = x.v_cache.reshape(case.B * nb, page, case.Hkv, case.d)
        table = perm.view(case.B, nb).to(torch.int32).contiguous().cuda()
        fa.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table, lens, num_splits=splits, seqlens_k_host=x.lens,
                           workspace=gw.t, out=go.t, lse=gl.t)
    else:
        fa.fa_decode(q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), lens, num_splits=splits, seqlens_k_host=x.lens,
                     workspace=gw.t, out=go.t, lse=gl.t)
    go.assert_margins_intact("decode O")
    gl.assert_margins_intact("decode LSE")
    gw.assert_margins_intact("decode workspace")
    if nq == 1:
        rows = np.array([(b, h) for b in range(case.B) for h in range(case.Hq)], dtype=np.int32)
        ro, rl = oracle_decode_rows(x, rows)
        check(go.t.double().cpu().numpy().reshape(-1, case.d), gl.t.double().cpu().numpy().reshape(-1), ro, rl,
              "decode")
    else:
        assert torch.isfinite(go.t.float()).all() and not torch.isnan(gl.t).any()
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("rows,H,d,rd", [(1000, 2, 128, 64), (257, 40, 128, 120)])  # narrow and wide rows
def test_rope_writes_stay_inside_its_tensor(rows, H, d, rd):
    import flashattention_forward_fa_gb300 as fa
    g = torch.Generator("cpu").manual_seed(912)
    x = torch.randn(rows, H, d, generator=g).to(torch.bfloat16)
    gx = Guarded((rows, H, d), torch.bfloat16, 4096)
    gx.t.copy_(x.cuda())
    pos = torch.arange(rows, dtype=torch.int32, device="cuda")
    fa.fa_rope(gx.t, pos, fa.rope_tables(rows, rd, device="cuda"))
    gx.assert_margins_intact("fa_rope")
    assert torch.equal(gx.t[..., rd:].cpu(), x[..., rd:])
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("cu_q,cu_k,max_q,max_k", [
    ([0, 40, 230], [0, 40, 100], 256, 256),       # the last query sequence runs past total_q = 100
    ([0, 60, 50, 100], [0, 30, 60, 100], 64, 64),  # decreasing query offsets
    ([0, 90, 100], [0, 50, 100], 64, 64),          # a sequence longer than max_seqlen_q
    ([0, 40, 100], [0, 40, 170], 128, 256),        # key offsets past total_k = 100
], ids=["past_total_q", "decreasing", "longer_than_max", "keys_past_total_k"])
def test_inconsistent_device_cu_seqlens_are_reported_not_written(cu_q, cu_k, max_q, max_k):
    # No host copy is passed, so only the kernel's own check stands between these offsets and the
    # plain stores.  The outputs sit in sentinel margins wider than any offset here reaches, so
    # even a failed check could only write into memory the test owns.
    import flashattention_forward_fa_gb300 as fa
    total_q, total_k, Hq, Hkv, d = 100, 100, 2, 2, 64
    g = torch.Generator("cpu").manual_seed(913)
    q = torch.randn(total_q, Hq, d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(total_k, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(total_k, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    go = Guarded((total_q, Hq, d), torch.bfloat16, 256 * Hq * d)
    gl = Guarded((Hq, total_q), torch.float32, 1024)
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    fa.fa_device_status(clear=True)
    fa.fa_fwd_varlen(q, k, v, cq, ck, max_q, max_k, causal=True, out=go.t, lse=gl.t)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) & 2
    go.assert_margins_intact("O")
    gl.assert_margins_intact("LSE")
