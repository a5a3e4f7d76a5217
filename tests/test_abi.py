"""CPU-side checks of the C ABI: the library builds/loads, exports every symbol
declared in include/fa.h, and rejects bad arguments on the host before any
CUDA call.  No compute runs here (there is no GPU)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    from flashattention_forward_fa_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_entry_points():
    syms = declared_symbols()
    for name in ("fa_fwd", "fa_fwd_varlen", "fa_decode", "fa_decode_workspace_size", "fa_decode_max_splits",
                 "fa_last_error", "fa_device_status"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    from flashattention_forward_fa_gb300 import build
    out = subprocess.check_output(["nm", "-D", "--defined-only", build.LIB]).decode()
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    for name in declared_symbols():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_no_cpu_fallback_symbols(lib):
    # the product library carries no host implementation of the attention math:
    # every compute entry point launches kernels, nothing links the oracle
    from flashattention_forward_fa_gb300 import build
    out = subprocess.check_output(["nm", "-D", build.LIB]).decode()
    assert "oracle" not in out


def _binding():
    import flashattention_forward_fa_gb300 as fa
    from flashattention_forward_fa_gb300 import _binding as b
    b.load_library()
    return fa, b


def test_invalid_arguments_rejected_on_host(lib):
    _, b = _binding()
    L = b.load_library()
    dummy = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails first
    # null q
    assert L.fa_fwd(None, dummy, dummy, dummy, None, 1, 2, 2, 8, 8, 64, 0.125, 0, 0, None, None, None) == 1
    assert b"non-null" in L.fa_last_error()
    # Hq % Hkv != 0
    assert L.fa_fwd(dummy, dummy, dummy, dummy, None, 1, 6, 4, 8, 8, 64, 0.125, 0, 0, None, None, None) == 1
    assert b"multiple" in L.fa_last_error()
    # unsupported head dim
    assert L.fa_fwd(dummy, dummy, dummy, dummy, None, 1, 2, 2, 8, 8, 96, 0.125, 0, 0, None, None, None) == 2
    # scale <= 0
    assert L.fa_fwd(dummy, dummy, dummy, dummy, None, 1, 2, 2, 8, 8, 64, 0.0, 0, 0, None, None, None) == 1
    # non-positive sizes
    assert L.fa_fwd(dummy, dummy, dummy, dummy, None, 0, 2, 2, 8, 8, 64, 0.1, 0, 0, None, None, None) == 1
    assert L.fa_fwd(dummy, dummy, dummy, dummy, None, 1, 2, 2, 0, 8, 64, 0.1, 0, 0, None, None, None) == 1
    # misaligned pointer
    odd = ctypes.c_void_p(0x1002)
    assert L.fa_fwd(odd, dummy, dummy, dummy, None, 1, 2, 2, 8, 8, 64, 0.1, 0, 0, None, None, None) == 1
    assert b"aligned" in L.fa_last_error()


def test_varlen_host_cu_seqlens_checked(lib):
    _, b = _binding()
    L = b.load_library()
    dummy = ctypes.c_void_p(0x1000)
    IntArr = ctypes.c_int * 4
    bad_start = IntArr(1, 3, 5, 8)
    assert L.fa_fwd_varlen(dummy, dummy, dummy, dummy, None, 3, 2, 2, 8, 8, 8, 8, 64, 0.1, 0, 0, dummy, dummy,
                           ctypes.cast(bad_start, b._ip), None) == 1
    non_mono = IntArr(0, 5, 3, 8)
    assert L.fa_fwd_varlen(dummy, dummy, dummy, dummy, None, 3, 2, 2, 8, 8, 8, 8, 64, 0.1, 0, 0, dummy, dummy,
                           ctypes.cast(non_mono, b._ip), None) == 1
    assert b"non-decreasing" in L.fa_last_error()
    wrong_total = IntArr(0, 3, 5, 7)
    assert L.fa_fwd_varlen(dummy, dummy, dummy, dummy, None, 3, 2, 2, 8, 8, 8, 8, 64, 0.1, 0, 0, dummy, dummy,
                           ctypes.cast(wrong_total, b._ip), None) == 1
    too_long = IntArr(0, 6, 7, 8)
    assert L.fa_fwd_varlen(dummy, dummy, dummy, dummy, None, 3, 2, 2, 8, 8, 4, 8, 64, 0.1, 0, 0, dummy, dummy,
                           ctypes.cast(too_long, b._ip), None) == 1
    # null cu_seqlens
    assert L.fa_fwd_varlen(dummy, dummy, dummy, dummy, None, 3, 2, 2, 8, 8, 8, 8, 64, 0.1, 0, 0, None, dummy,
                           None, None) == 1


def test_decode_arguments_checked(lib):
    _, b = _binding()
    L = b.load_library()
    dummy = ctypes.c_void_p(0x1000)
    # null seqlens
    assert L.fa_decode(dummy, dummy, dummy, dummy, None, 2, 8, 2, 64, 128, 0.1, 0, None, None, 0, dummy, 1 << 20,
                       None) == 1
    # negative num_splits
    assert L.fa_decode(dummy, dummy, dummy, dummy, None, 2, 8, 2, 64, 128, 0.1, 0, dummy, None, -1, dummy,
                       1 << 20, None) == 1


def test_workspace_size_formula(lib):
    _, b = _binding()
    L = b.load_library()
    assert L.fa_decode_workspace_size(64, 32, 128, 9) == 64 * 32 * 9 * 129 * 4
    assert L.fa_decode_workspace_size(0, 32, 128, 9) == 0


def test_decode_split_plan_bounds(lib):
    _, b = _binding()
    L = b.load_library()
    # explicit split count: chunk = ceil(longest / n) rounded up to 64
    lens = (ctypes.c_int * 3)(100, 1000, 640)
    assert L.fa_decode_max_splits(3, 8, 2, 1024, 0, ctypes.cast(lens, b._ip), 4) == 4
    # one split when asked for one
    assert L.fa_decode_max_splits(3, 8, 2, 1024, 0, ctypes.cast(lens, b._ip), 1) == 1
    # window caps the key range
    assert L.fa_decode_max_splits(3, 8, 2, 1024, 64, None, 8) == 1
    assert L.fa_decode_max_splits(0, 8, 2, 1024, 0, None, 0) == 0


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    fa, b = _binding()
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(b.FAError):
        fa.fa_fwd(q, q, q)


def test_paged_decode_arguments_checked(lib):
    _, b = _binding()
    L = b.load_library()
    d = ctypes.c_void_p(0x1000)
    args = lambda **kw: [kw.get("q", d), d, d, d, None, 2, 8, 2, kw.get("num_pages", 10), kw.get("page", 64), 128,
                         ctypes.c_float(0.1), 0, kw.get("table", d), kw.get("max_blocks", 4), kw.get("lens", d), None,
                         0, d, 1 << 24, None]
    assert L.fa_decode_paged(*args(page=96)) == 1            # not a multiple of 64
    assert b"multiple of 64" in L.fa_last_error()
    assert L.fa_decode_paged(*args(page=0)) == 1
    assert L.fa_decode_paged(*args(table=None)) == 1
    assert L.fa_decode_paged(*args(lens=None)) == 1
    assert L.fa_decode_paged(*args(num_pages=0)) == 1
    assert L.fa_decode_paged(*args(max_blocks=0)) == 1


def test_ex_entry_points_read_their_structs(lib):
    # the ctypes mirrors of fa_fwd_args / fa_decode_args line up with the C layout: each field
    # checked here is read from its own offset and triggers its own host-side error
    _, b = _binding()
    L = b.load_library()
    d = 0x1000
    a = b.FwdArgs(q=d, k=d, v=d, o=d, B=1, Hq=6, Hkv=4, Nq=8, Nk=8, d=64, scale=0.1)
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 1 and b"multiple" in L.fa_last_error()
    a = b.FwdArgs(q=d, k=d, v=d, o=d, B=1, Hq=2, Hkv=2, Nq=8, Nk=8, d=96, scale=0.1)
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 2
    a = b.FwdArgs(q=d, k=d, v=d, o=d, B=1, Hq=2, Hkv=2, Nq=8, Nk=8, d=64, scale=0.1, alibi_slopes=0x1002)
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 1 and b"alibi" in L.fa_last_error()
    a = b.FwdArgs(q=d, k=d, v=d, o=d, B=1, Hq=2, Hkv=2, Nq=8, Nk=8, d=64, scale=0.1, cu_seqlens_q=d)
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 1 and b"cu_seqlens" in L.fa_last_error()
    x = b.DecodeArgs(q=d, k=d, v=d, o=d, B=2, Hq=8, Hkv=2, d=128, scale=0.1, Ncap=64, seqlens_k=d,
                     block_table=d, page_size=96, num_pages=4, max_blocks=2)
    assert L.fa_decode_ex(ctypes.byref(x), None) == 1 and b"multiple of 64" in L.fa_last_error()
    x = b.DecodeArgs(q=d, k=d, v=d, o=d, B=2, Hq=8, Hkv=2, d=128, scale=0.1, Ncap=64, num_splits=-1, seqlens_k=d)
    assert L.fa_decode_ex(ctypes.byref(x), None) == 1 and b"num_splits" in L.fa_last_error()


def test_alibi_slope_schedule():
    _, b = _binding()
    s8 = b.alibi_slopes(8)
    assert s8 == [2.0 ** -(i + 1) for i in range(8)]
    s12 = b.alibi_slopes(12)
    assert s12[:8] == s8 and s12[8:] == [2.0 ** -(0.5 + i) for i in range(4)]


def test_rope_arguments_checked(lib):
    # fa_fwd_args' rope fields sit after alibi_slopes and each is validated on the host
    _, b = _binding()
    L = b.load_library()
    d = 0x1000
    base = dict(q=d, k=d, v=d, o=d, B=1, Hq=2, Hkv=2, Nq=8, Nk=8, d=64, scale=0.1)
    a = b.FwdArgs(**base, rope_cos=d)                                   # sin missing
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 1 and b"rope_sin" in L.fa_last_error()
    a = b.FwdArgs(**base, rope_cos=d, rope_sin=d, rope_rows=16, rope_dim=12)
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 1 and b"rope_dim" in L.fa_last_error()
    a = b.FwdArgs(**base, rope_cos=d, rope_sin=d, rope_rows=16, rope_dim=128)   # > d
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 1 and b"rope_dim" in L.fa_last_error()
    a = b.FwdArgs(**base, rope_cos=d, rope_sin=d, rope_rows=0, rope_dim=64)
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 1 and b"rope_rows" in L.fa_last_error()
    a = b.FwdArgs(**base, rope_cos=d + 4, rope_sin=d, rope_rows=16, rope_dim=64)
    assert L.fa_fwd_ex(ctypes.byref(a), None) == 1 and b"aligned" in L.fa_last_error()
    # fa_rope(x, rows, heads, d, rotary_dim, positions, cos, sin, table_rows, stream)
    L.fa_rope.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert L.fa_rope(None, 4, 2, 64, 64, d, d, d, 8, None) == 1
    assert L.fa_rope(d, 4, 2, 64, 60, d, d, d, 8, None) == 1 and b"rotary_dim" in L.fa_last_error()
    assert L.fa_rope(d, 4, 2, 64, 72, d, d, d, 8, None) == 1
    assert L.fa_rope(d, -1, 2, 64, 64, d, d, d, 8, None) == 1
    assert L.fa_rope(d, 4, 2, 64, 64, d, d + 8, d, 8, None) == 1 and b"aligned" in L.fa_last_error()
    assert L.fa_rope(d, 0, 2, 64, 64, d, d, d, 8, None) == 0                  # nothing to do
    assert L.fa_rope(d, 4, 2, 2048, 1032, d, d, d, 8, None) == 2 and b"1024" in L.fa_last_error()
    assert L.fa_rope(d, 4, 1 << 20, 4096, 64, d, d, d, 8, None) == 1 and b"31 bits" in L.fa_last_error()


def test_rope_tables_match_oracle_tables():
    # the binding's table helper builds the same angles as the oracle's (both from
    # p * base^(-2i / rotary_dim)); fp32 rounding of the fp64 values is the only difference
    import numpy as np
    from oracle import rope as orope
    _, b = _binding()
    c, s = b.rope_tables(300, 64, device="cpu")
    rc, rs = orope.tables(300, 64)
    assert c.dtype.is_floating_point and tuple(c.shape) == (300, 32)
    np.testing.assert_allclose(c.numpy(), rc, atol=1e-7)
    np.testing.assert_allclose(s.numpy(), rs, atol=1e-7)


def test_selftest_wait_timeout_arguments_checked(lib):
    _, b = _binding()
    L = b.load_library()
    assert L.fa_selftest_wait_timeout(0, None) == 1
    assert L.fa_selftest_wait_timeout(5000, None) == 1 and b"limit_ms" in L.fa_last_error()


def test_selftest_prefill_abort_arguments_checked(lib):
    _, b = _binding()
    L = b.load_library()
    a = b.FwdArgs()
    assert L.fa_selftest_prefill_abort(ctypes.byref(a), 0, None) == 1 and b"v_loads" in L.fa_last_error()
    assert L.fa_selftest_prefill_abort(None, 2, None) == 1 and b"non-null" in L.fa_last_error()
    # otherwise the arguments go through the same checks as fa_fwd_ex (here: null tensors)
    assert L.fa_selftest_prefill_abort(ctypes.byref(a), 2, None) == 1


def test_host_int_arrays_reach_the_library_by_address():
    """A host int32 copy (cu_seqlens_q_host, seqlens_k_host) is handed to the C ABI as an address:
    a contiguous int32 CPU tensor or numpy array without a copy, any other sequence copied into a
    ctypes array that the caller keeps alive; the address reads back the same values."""
    import numpy as np
    import torch
    _, b = _binding()
    vals = [0, 5, 17, 300, 301, 1024]
    t = torch.tensor(vals, dtype=torch.int32)
    a = np.array(vals, dtype=np.int32)
    for src, no_copy in ((t, True), (a, True), (vals, False), (torch.tensor(vals), False), (np.array(vals), False)):
        h = b._host_ints(src)
        addr = b._host_ptr(h)
        assert isinstance(addr, int) and addr != 0
        got = list((ctypes.c_int * len(vals)).from_address(addr))
        assert got == vals, (type(src), got)
        if no_copy:
            expect = src.data_ptr() if isinstance(src, torch.Tensor) else src.__array_interface__["data"][0]
            assert addr == expect
    assert b._host_ints(None) is None and b._host_ptr(None) is None
