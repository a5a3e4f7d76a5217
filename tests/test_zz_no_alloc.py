"""Decode with no device allocation (fa_decode_noalloc, through the C ABI).

Some callers of this library cannot call cudaMalloc — a plugin inside an
inference engine that is handed only its input and output buffers, or a
serving loop that must not take the allocator's locks or the device
synchronisation an allocation can cause.  fa_decode_noalloc serves them: its
split-KV partials live in a fixed scratch array inside the library instead of
a caller workspace.  This file checks it against the ordinary fa_decode (with
a caller-owned workspace) and against the fp64 oracle on two calls in a row
with different inputs, so a stale scratch from the first call would show in
the second; runs the largest problem the scratch is documented to hold
(B=64, Hq=32, d=128 with 15 splits) against the oracle; and checks that
problems too large for the scratch are refused before any launch, with real
device buffers so that nothing could fault even if a check regressed.

The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from fa_workloads import DECODE_CACHE, DecodeCase, make_decode
from tests._util import check, oracle_decode_rows

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_INVALID = 0, 1


def _lib():
    from flashattention_forward_fa_gb300 import _binding
    return _binding, _binding.load_library()


def _noalloc_through_abi(lib, b, x, dq, dk, dv, lens_dev, o, lse, num_splits=0):
    c = x.case
    host = (ctypes.c_int * c.B)(*x.lens)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fa_decode_noalloc(
        ctypes.c_void_p(dq.data_ptr()), ctypes.c_void_p(dk.data_ptr()), ctypes.c_void_p(dv.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), c.B, c.Hq, c.Hkv, c.Ncap, c.d,
        ctypes.c_float(c.softmax_scale), c.window, ctypes.c_void_p(lens_dev.data_ptr()),
        ctypes.cast(host, b._ip), num_splits, stream)


def _all_pairs(B, Hq):
    return np.array([(b, h) for b in range(B) for h in range(Hq)], dtype=np.int32)


def _oracle_check(x, o, lse, what):
    c = x.case
    ro, rl = oracle_decode_rows(x, _all_pairs(c.B, c.Hq))
    return check(o.double().cpu().numpy().reshape(-1, c.d), lse.double().cpu().numpy().reshape(-1), ro, rl, what)


CASES = [
    DecodeCase("noalloc_first", B=6, Hq=16, Hkv=4, Ncap=3000, d=128, lens=[3000, 1, 64, 1500, 777, 2048], seed=61),
    DecodeCase("noalloc_second", B=5, Hq=8, Hkv=2, Ncap=900, d=64, lens=[13, 900, 450, 129, 2], seed=62),
]


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row():
    import flashattention_forward_fa_gb300 as fa
    b, lib = _lib()
    for case in CASES:
        x = make_decode(case)
        dq, dk, dv = x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda()
        lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
        # the existing entry point, with a workspace the caller allocates
        ref_o, ref_l = fa.fa_decode(dq, dk, dv, lens, scale=case.softmax_scale, seqlens_k_host=x.lens)
        # the no-allocation entry point: outputs pre-allocated by the test, no workspace
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        assert _noalloc_through_abi(lib, b, x, dq, dk, dv, lens, o, lse) == FA_OK, lib.fa_last_error()
        torch.cuda.synchronize()
        check(o.double().cpu().numpy().reshape(-1, case.d), lse.double().cpu().numpy().reshape(-1),
              ref_o.double().cpu().numpy().reshape(-1, case.d), ref_l.double().cpu().numpy().reshape(-1),
              case.name)
        _oracle_check(x, o, lse, case.name + " vs oracle")
    assert fa.fa_device_status() == 0


def test_noalloc_at_its_documented_bound_and_one_split_past_it():
    # decode_cache's shape (B=64, Hq=32, Hkv=8, d=128) with 15 splits: 64*32*15*129*4 = 15.85 MB of
    # partials, the largest split count the 16 MiB scratch holds at this shape; 16 splits need
    # 16.9 MB and must be refused before any launch (the outputs stay as they were).  Its lengths,
    # with the first sequence at the full 8192 slots so that the plan uses exactly the split count
    # asked for (8192 keys in 15 chunks of 576, or 16 of 512).
    import flashattention_forward_fa_gb300 as fa
    b, lib = _lib()
    x = make_decode(DECODE_CACHE)
    x.lens = [8192] + list(x.lens[1:])
    c = x.case
    dq, dk, dv = x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda()
    lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
    assert fa.fa_decode_max_splits(c.B, c.Hq, c.Hkv, c.Ncap, 0, x.lens, 15) == 15
    o = torch.full((c.B, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc_through_abi(lib, b, x, dq, dk, dv, lens, o, lse, num_splits=15) == FA_OK, lib.fa_last_error()
    torch.cuda.synchronize()
    res = _oracle_check(x, o, lse, "noalloc 15 splits vs oracle")
    assert res["rows"] == c.B * c.Hq
    o2 = torch.full_like(o, 7.0)
    l2 = torch.full_like(lse, 7.0)
    assert fa.fa_decode_max_splits(c.B, c.Hq, c.Hkv, c.Ncap, 0, x.lens, 16) == 16
    assert _noalloc_through_abi(lib, b, x, dq, dk, dv, lens, o2, l2, num_splits=16) == FA_ERR_INVALID
    assert b"built-in scratch" in lib.fa_last_error()
    torch.cuda.synchronize()
    assert torch.all(o2 == 7.0) and torch.all(l2 == 7.0)
    assert fa.fa_device_status() == 0


def test_noalloc_refuses_problems_larger_than_its_scratch():
    # B=64, Hq=64, d=128 with 64 splits needs 64*64*64*129*4 B = 135 MB of partials > 16 MiB.  The
    # buffers are real (a 67 MB cache with one KV head), so a regressed size check could not make
    # the kernels touch memory that is not there.
    import flashattention_forward_fa_gb300 as fa
    b, lib = _lib()
    case = DecodeCase("noalloc_too_big", B=64, Hq=64, Hkv=1, Ncap=4096, d=128, lens=[4096] * 64, seed=63)
    q = torch.zeros((case.B, case.Hq, case.d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((case.B, case.Ncap, case.Hkv, case.d), dtype=torch.bfloat16, device="cuda")
    lens = torch.full((case.B,), 4096, dtype=torch.int32, device="cuda")
    o = torch.full((case.B, case.Hq, case.d), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((case.B, case.Hq), 3.0, dtype=torch.float32, device="cuda")

    class _X:
        pass
    x = _X()
    x.case, x.lens = case, case.lens
    st = _noalloc_through_abi(lib, b, x, q, kc, kc, lens, o, lse, num_splits=64)
    assert st == FA_ERR_INVALID
    assert b"built-in scratch" in lib.fa_last_error()
    torch.cuda.synchronize()
    assert torch.all(o == 3.0) and torch.all(lse == 3.0)
    assert fa.fa_device_status() == 0
