"""GB300 (sm_103a) fused attention forward: Python binding over libfa_gb300.so.

Argument marshalling only — every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/fa.h``.  PyTorch supplies device
memory and streams.  There is no CPU fallback: when the library is missing or
the device is not sm_103, calls raise.

Entry points (same names as the C ABI):

* ``fa_fwd(q, k, v, ...)``         padded-batch prefill   q [B, Nq, Hq, d]
* ``fa_fwd_varlen(q, k, v, ...)``  packed varlen prefill  q [total_q, Hq, d]
* ``fa_decode(q, k_cache, v_cache, seqlens_k, ...)``  one new token per sequence
* ``fa_decode_paged(...)``         decode over a paged (block-table) KV cache
* ``fa_decode_noalloc(...)``       the same decode with no device allocation at all
* ``fa_rope(x, positions, (cos, sin))``  rotary embedding in place (K before the
  fused prefill, or a KV cache); ``rope_tables`` builds the usual tables
* ``fa_fwd_ex`` / ``fa_decode_ex`` (C ABI): every option in one struct; reached from
  the wrappers above when ``alibi_slopes`` or ``rope`` is given
* ``fa_device_status()``           read/clear the kernels' error word
* ``fa_selftest_wait_timeout()``   a wait that runs out on purpose, ending with the timeout bit
* ``fa_selftest_prefill_abort()``  a prefill whose V loads stop on purpose: its abort path runs
"""

from __future__ import annotations

from ._binding import (  # noqa: F401
    DecodeArgs,
    FAError,
    FwdArgs,
    alibi_slopes,
    decode_workspace_size,
    fa_decode,
    fa_decode_max_splits,
    fa_decode_noalloc,
    fa_decode_paged,
    fa_device_status,
    fa_fwd,
    fa_fwd_varlen,
    fa_rope,
    fa_selftest_prefill_abort,
    fa_selftest_wait_timeout,
    library_path,
    load_library,
    rope_tables,
)

__all__ = [
    "FAError",
    "FwdArgs",
    "DecodeArgs",
    "alibi_slopes",
    "fa_fwd",
    "fa_fwd_varlen",
    "fa_rope",
    "rope_tables",
    "fa_decode",
    "fa_decode_max_splits",
    "fa_decode_noalloc",
    "fa_decode_paged",
    "decode_workspace_size",
    "fa_device_status",
    "fa_selftest_wait_timeout",
    "fa_selftest_prefill_abort",
    "load_library",
    "library_path",
]
