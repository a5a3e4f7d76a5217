"""Decode with no device allocation (fa_decode_noalloc, through the C ABI).

Some callers of this library cannot call cudaMalloc — a plugin inside an
inference engine that is handed only its input and output buffers, or a
serving loop that must not take the allocator's locks or the device
synchronisation an allocation can cause.  fa_decode_noalloc serves them: its
split-KV partials live in a fixed scratch array inside the library instead of
a caller workspace.  This file checks it against the ordinary fa_decode (with
a caller-owned workspace) on two calls in a row with different inputs, so a
stale scratch from the first call would show in the second, and checks that
a problem too large for the scratch is refused before any launch.

The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from fa_workloads import DecodeCase, make_decode
from tests._util import check

pytestmark = pytest.mark.gpu

FA_ERR_INVALID = 1


def _lib():
    from flashattention_forward_fa_gb300 import _binding
    return _binding, _binding.load_library()


def _noalloc_through_abi(lib, b, x, lens_dev, o, lse, num_splits=0):
    c = x.case
    host = (ctypes.c_int * c.B)(*x.lens)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fa_decode_noalloc(
        ctypes.c_void_p(x._dq.data_ptr()), ctypes.c_void_p(x._dk.data_ptr()), ctypes.c_void_p(x._dv.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), c.B, c.Hq, c.Hkv, c.Ncap, c.d,
        ctypes.c_float(c.softmax_scale), c.window, ctypes.c_void_p(lens_dev.data_ptr()),
        ctypes.cast(host, b._ip), num_splits, stream)


CASES = [
    DecodeCase("noalloc_first", B=6, Hq=16, Hkv=4, Ncap=3000, d=128, lens=[3000, 1, 64, 1500, 777, 2048], seed=61),
    DecodeCase("noalloc_second", B=5, Hq=8, Hkv=2, Ncap=900, d=64, lens=[13, 900, 450, 129, 2], seed=62),
]


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row():
    import flashattention_forward_fa_gb300 as fa
    b, lib = _lib()
    for case in CASES:
        x = make_decode(case)
        x._dq, x._dk, x._dv = x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda()
        lens = torch.tensor(x.lens, dtype=torch.int32, device="cuda")
        # the existing entry point, with a workspace the caller allocates
        ref_o, ref_l = fa.fa_decode(x._dq, x._dk, x._dv, lens, scale=case.softmax_scale, seqlens_k_host=x.lens)
        # the no-allocation entry point: outputs pre-allocated by the test, no workspace
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        assert _noalloc_through_abi(lib, b, x, lens, o, lse) == 0, lib.fa_last_error()
        torch.cuda.synchronize()
        check(o.double().cpu().numpy().reshape(-1, case.d), lse.double().cpu().numpy().reshape(-1),
              ref_o.double().cpu().numpy().reshape(-1, case.d), ref_l.double().cpu().numpy().reshape(-1),
              case.name)
    assert fa.fa_device_status() == 0


def test_noalloc_refuses_problems_larger_than_its_scratch():
    b, lib = _lib()
    # B=64, Hq=64, d=128 with 64 splits needs 64*64*64*129*4 B = 135 MB of partials > 16 MiB
    lens = (ctypes.c_int * 64)(*([8192] * 64))
    dummy = ctypes.c_void_p(0x100000)   # never dereferenced: the size check fails first
    st = lib.fa_decode_noalloc(dummy, dummy, dummy, dummy, None, 64, 64, 8, 8192, 128, ctypes.c_float(0.08), 0,
                               dummy, ctypes.cast(lens, b._ip), 64, None)
    assert st == FA_ERR_INVALID
    assert b"built-in scratch" in lib.fa_last_error()
