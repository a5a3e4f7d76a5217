"""ctypes binding of libfa_gb300.so (see include/fa.h for the contracts)."""

from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")
_lock = threading.Lock()
_lib = None

FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA", 4: "FA_ERR_TIMEOUT"}

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)

class FwdArgs(ctypes.Structure):
    """Mirror of fa_fwd_args (include/fa.h)."""
    _fields_ = [("q", _vp), ("k", _vp), ("v", _vp), ("o", _vp), ("lse", _vp),
                ("B", _i), ("Hq", _i), ("Hkv", _i), ("Nq", _i), ("Nk", _i), ("d", _i),
                ("scale", _f), ("causal", _i), ("window", _i),
                ("seqlens_q", _vp), ("seqlens_k", _vp), ("cu_seqlens_q", _vp), ("cu_seqlens_k", _vp),
                ("total_q", _i), ("total_k", _i), ("cu_seqlens_q_host", _vp), ("alibi_slopes", _vp),
                ("rope_cos", _vp), ("rope_sin", _vp), ("rope_rows", _i), ("rope_dim", _i)]


class DecodeArgs(ctypes.Structure):
    """Mirror of fa_decode_args (include/fa.h)."""
    _fields_ = [("q", _vp), ("k", _vp), ("v", _vp), ("o", _vp), ("lse", _vp),
                ("B", _i), ("Hq", _i), ("Hkv", _i), ("d", _i), ("scale", _f), ("window", _i), ("Ncap", _i),
                ("block_table", _vp), ("max_blocks", _i), ("page_size", _i), ("num_pages", _i),
                ("seqlens_k", _vp), ("seqlens_k_host", _vp), ("num_splits", _i),
                ("workspace", _vp), ("workspace_bytes", _sz), ("alibi_slopes", _vp), ("Nq", _i)]


_SIGS = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _vp, _vp]),
    "fa_fwd_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _vp, _vp,
                           _vp]),
    "fa_decode_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _i, _vp, _sz, _vp]),
    "fa_decode_max_splits": (_i, [_i, _i, _i, _i, _i, _vp, _i]),
    "fa_decode_paged": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _vp, _i, _vp,
                             _sz, _vp]),
    "fa_fwd_ex": (_i, [ctypes.POINTER(FwdArgs), _vp]),
    "fa_decode_ex": (_i, [ctypes.POINTER(DecodeArgs), _vp]),
    "fa_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _i, _vp]),
    "fa_rope": (_i, [_vp, ctypes.c_longlong, _i, _i, _i, _vp, _vp, _vp, _i, _vp]),
    "fa_selftest_wait_timeout": (_i, [_i, _vp]),
    "fa_selftest_prefill_abort": (_i, [ctypes.POINTER(FwdArgs), _i, _vp]),
    "fa_last_error": (ctypes.c_char_p, []),
    "fa_device_status": (_i, [ctypes.POINTER(ctypes.c_uint32), _i]),
}


class FAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_NAMES.get(status, status)}: {msg}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libfa_gb300.so (raises if it has not been built)."""
    global _lib
    lib = _lib
    if lib is not None:  # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise FAError(FA_ERR_UNSUPPORTED,
                              f"{_LIB_PATH} is missing; build it with "
                              "`python -m flashattention_forward_fa_gb300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int):
    if status != FA_OK:
        raise FAError(status, load_library().fa_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t: torch.Tensor):
    # The raw handle of torch's current stream on t's device (the fast accessor when present).
    if _raw_stream is not None:
        return _raw_stream(t.device.index)
    return torch.cuda.current_stream(t.device).cuda_stream


def _host_ints(x):
    """A host int32 array for the C ABI: None, a contiguous int32 CPU tensor or numpy array (passed
    by address, no copy), or any sequence of ints (copied into a ctypes array, which the caller
    keeps alive until the call returns)."""
    if x is None:
        return None
    if isinstance(x, torch.Tensor) and not x.is_cuda and x.dtype == torch.int32 and x.is_contiguous():
        return x.data_ptr()
    if isinstance(x, np.ndarray) and x.dtype == np.int32 and x.flags["C_CONTIGUOUS"]:
        return x.__array_interface__["data"][0]
    vals = [int(v) for v in (x.tolist() if isinstance(x, (torch.Tensor, np.ndarray)) else x)]
    return (ctypes.c_int * len(vals))(*vals)


def _host_ptr(h):
    """The address (or None) of what _host_ints returned, for a void* argument."""
    if h is None or isinstance(h, int):
        return h
    return ctypes.addressof(h)


def alibi_slopes(num_heads: int) -> list:
    """The geometric ALiBi slope schedule of Press et al. (ALiBi paper): for n heads, n a power
    of two, slopes 2^(-8/n), 2^(-16/n), ..., 2^(-8); otherwise the schedule of the largest power
    of two below n followed by every other slope of the schedule for twice that power.  The
    source pages give no slopes; this is the usual choice, offered for convenience."""
    def pow2(n):
        return [2.0 ** (-8.0 * (i + 1) / n) for i in range(n)]
    if num_heads <= 0:
        return []
    p2 = 1 << (num_heads.bit_length() - 1)
    if p2 == num_heads:
        return pow2(num_heads)
    return pow2(p2) + pow2(2 * p2)[0::2][: num_heads - p2]


def _slopes_ptr(alibi_slopes, Hq: int, device):
    if alibi_slopes is None:
        return None, None
    t = alibi_slopes if isinstance(alibi_slopes, torch.Tensor) else torch.tensor(alibi_slopes, dtype=torch.float32)
    t = t.to(device=device, dtype=torch.float32).contiguous()
    if t.numel() != Hq:
        raise FAError(FA_ERR_INVALID, "alibi_slopes needs one slope per query head")
    return t, t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=torch.bfloat16):
    if isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.is_contiguous():
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise FAError(FA_ERR_INVALID, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise FAError(FA_ERR_INVALID, f"{name} must be {dtype}")
    raise FAError(FA_ERR_INVALID, f"{name} must be contiguous")


def rope_tables(max_pos: int, rotary_dim: int, base: float = 10000.0, device="cuda"):
    """The usual RoPE tables: angle p * base^(-2i / rotary_dim) for position p < max_pos and pair
    i < rotary_dim / 2, as fp32 (cos, sin) tensors [max_pos, rotary_dim / 2] on `device`.  A setup
    step run once per model (the tables are an input of fa_rope and of the fused prefill)."""
    i = torch.arange(rotary_dim // 2, dtype=torch.float64)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * (base ** (-2.0 * i / rotary_dim))[None, :]
    return (torch.cos(ang).to(torch.float32).contiguous().to(device),
            torch.sin(ang).to(torch.float32).contiguous().to(device))


def _check_tables(rope, rotary_dim: Optional[int], d: int):
    if not (isinstance(rope, (tuple, list)) and len(rope) == 2):
        raise FAError(FA_ERR_INVALID, "rope must be a (cos, sin) pair of tables")
    cos_t, sin_t = rope
    _need(cos_t, "rope cos", torch.float32)
    _need(sin_t, "rope sin", torch.float32)
    if cos_t.dim() != 2 or cos_t.shape != sin_t.shape:
        raise FAError(FA_ERR_INVALID, "rope tables must both be [positions, rotary_dim / 2]")
    rd = int(rotary_dim) if rotary_dim is not None else 2 * cos_t.shape[1]
    if rd <= 0 or rd > d or 2 * cos_t.shape[1] != rd:
        raise FAError(FA_ERR_INVALID, f"rope tables have {cos_t.shape[1]} pairs, rotary_dim is {rd}, d is {d}")
    return cos_t, sin_t, rd


def _set_rope(a: FwdArgs, rope, rotary_dim: Optional[int], d: int):
    if rope is None:
        return
    cos_t, sin_t, rd = _check_tables(rope, rotary_dim, d)
    a.rope_cos, a.rope_sin, a.rope_rows, a.rope_dim = _ptr(cos_t), _ptr(sin_t), cos_t.shape[0], rd


def fa_rope(x: torch.Tensor, positions: torch.Tensor, rope, rotary_dim: Optional[int] = None) -> torch.Tensor:
    """Rotate x in place: x bf16 [..., H, d], positions int32 with one entry per row of the
    leading dims, rope = (cos, sin) tables [max_pos, rotary_dim / 2].  Returns x."""
    lib = load_library()
    _need(x, "x")
    _need(positions, "positions", torch.int32)
    if x.dim() < 2:
        raise FAError(FA_ERR_INVALID, "x must be [..., H, d]")
    H, d = x.shape[-2], x.shape[-1]
    rows = x.numel() // (H * d) if x.numel() else 0
    if positions.numel() != rows:
        raise FAError(FA_ERR_INVALID, f"positions has {positions.numel()} entries for {rows} rows")
    cos_t, sin_t, rd = _check_tables(rope, rotary_dim, d)
    _check(lib.fa_rope(_ptr(x), rows, H, d, rd, _ptr(positions), _ptr(cos_t), _ptr(sin_t), cos_t.shape[0],
                       _stream(x)))
    return x


def fa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False, window: int = 0,
           scale: Optional[float] = None, seqlens_q: Optional[torch.Tensor] = None,
           seqlens_k: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None, return_lse: bool = True, alibi_slopes=None,
           rope=None, rotary_dim: Optional[int] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Padded-batch prefill.  q [B, Nq, Hq, d], k/v [B, Nk, Hkv, d] bf16 -> (O, LSE [B, Hq, Nq]).
    alibi_slopes: optional per-query-head slopes (bias -m_h |p - j| on the scaled scores).
    rope: optional (cos, sin) fp32 tables [positions, rotary_dim / 2]; the kernel rotates Q at
    position i + Lk - Lq after loading it.  K must already be rotated (fa_rope)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n)
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise FAError(FA_ERR_INVALID, "expected q [B,Nq,Hq,d] and k, v [B,Nk,Hkv,d]")
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    if k.shape[0] != B or k.shape[3] != d:
        raise FAError(FA_ERR_INVALID, "q and k disagree on B or d")
    for t, n in ((seqlens_q, "seqlens_q"), (seqlens_k, "seqlens_k")):
        if t is not None:
            _need(t, n, torch.int32)
    o = out if out is not None else torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    if alibi_slopes is None and rope is None:
        _check(lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d, sc,
                          int(bool(causal)), int(window), _ptr(seqlens_q), _ptr(seqlens_k), _stream(q)))
        return o, lse
    keep, sp = _slopes_ptr(alibi_slopes, Hq, q.device)
    a = FwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), o=_ptr(o), lse=_ptr(lse), B=B, Hq=Hq, Hkv=Hkv, Nq=Nq, Nk=Nk, d=d,
                scale=sc, causal=int(bool(causal)), window=int(window), seqlens_q=_ptr(seqlens_q),
                seqlens_k=_ptr(seqlens_k), alibi_slopes=sp)
    _set_rope(a, rope, rotary_dim, d)
    _check(lib.fa_fwd_ex(ctypes.byref(a), _stream(q)))
    return o, lse


def fa_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                  cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, causal: bool = False,
                  window: int = 0, scale: Optional[float] = None, cu_seqlens_q_host: Optional[Sequence[int]] = None,
                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  return_lse: bool = True, alibi_slopes=None, rope=None, rotary_dim: Optional[int] = None
                  ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Packed varlen prefill.  q [total_q, Hq, d], k/v [total_k, Hkv, d] -> (O, LSE [Hq, total_q]).
    alibi_slopes, rope, rotary_dim: as for fa_fwd (positions count from each sequence's start).
    cu_seqlens_q_host: optional host copy of cu_seqlens_q, checked before the launch; an int32 CPU
    tensor (or int32 numpy array) is passed by address, the cheapest form for a loop that calls
    this every step."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32)
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape:
        raise FAError(FA_ERR_INVALID, "expected q [total_q,Hq,d] and k, v [total_k,Hkv,d]")
    total_q, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    if B <= 0 or cu_seqlens_k.numel() != B + 1:
        raise FAError(FA_ERR_INVALID, "cu_seqlens_q/k must both have B + 1 entries")
    o = out if out is not None else torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    host = _host_ints(cu_seqlens_q_host)
    if alibi_slopes is not None or rope is not None:
        keep, sp = _slopes_ptr(alibi_slopes, Hq, q.device)
        a = FwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), o=_ptr(o), lse=_ptr(lse), B=B, Hq=Hq, Hkv=Hkv,
                    Nq=int(max_seqlen_q), Nk=int(max_seqlen_k), d=d, scale=sc, causal=int(bool(causal)),
                    window=int(window), cu_seqlens_q=_ptr(cu_seqlens_q), cu_seqlens_k=_ptr(cu_seqlens_k),
                    total_q=total_q, total_k=total_k,
                    cu_seqlens_q_host=_host_ptr(host), alibi_slopes=sp)
        _set_rope(a, rope, rotary_dim, d)
        _check(lib.fa_fwd_ex(ctypes.byref(a), _stream(q)))
        return o, lse
    _check(lib.fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, total_q, total_k,
                             int(max_seqlen_q), int(max_seqlen_k), d, sc, int(bool(causal)), int(window),
                             _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                             _host_ptr(host), _stream(q)))
    return o, lse


def decode_workspace_size(B: int, Hq: int, d: int, max_splits: int) -> int:
    return int(load_library().fa_decode_workspace_size(B, Hq, d, max_splits))


def fa_decode_max_splits(B: int, Hq: int, Hkv: int, Ncap: int, window: int = 0, seqlens_k_host=None,
                         num_splits: int = 0) -> int:
    host = _host_ints(seqlens_k_host)
    return int(load_library().fa_decode_max_splits(B, Hq, Hkv, Ncap, int(window),
                                                   _host_ptr(host),
                                                   int(num_splits)))


def fa_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seqlens_k: torch.Tensor,
              window: int = 0, scale: Optional[float] = None, num_splits: int = 0, seqlens_k_host=None,
              workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
              lse: Optional[torch.Tensor] = None, return_lse: bool = True, alibi_slopes=None
              ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Decode: q [B, Hq, d], caches [B, Ncap, Hkv, d], seqlens_k int32 [B] -> (O [B, Hq, d], LSE [B, Hq]).
    With q [B, Nq, Hq, d] the Nq new tokens are the last Nq cache slots (token t at position
    len - Nq + t, bottom-right causal) -> (O [B, Nq, Hq, d], LSE [B, Hq, Nq])."""
    lib = load_library()
    _need(q, "q")
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache")
    _need(seqlens_k, "seqlens_k", torch.int32)
    if q.dim() not in (3, 4) or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise FAError(FA_ERR_INVALID, "expected q [B,Hq,d] or [B,Nq,Hq,d] and caches [B,Ncap,Hkv,d]")
    B, Hq, d = q.shape[0], q.shape[-2], q.shape[-1]
    Nq = q.shape[1] if q.dim() == 4 else 1
    _, Ncap, Hkv, _ = k_cache.shape
    host = _host_ints(seqlens_k_host)
    hostp = _host_ptr(host)
    if workspace is None:
        S = lib.fa_decode_max_splits(B, Hq, Hkv, Ncap, int(window) + Nq - 1 if window > 0 else 0, hostp,
                                     int(num_splits))
        nbytes = lib.fa_decode_workspace_size(B * Nq, Hq, d, max(S, 1))
        workspace = torch.empty((nbytes + 3) // 4, dtype=torch.float32, device=q.device)
    o = out if out is not None else torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Nq) if q.dim() == 4 else (B, Hq), dtype=torch.float32, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    if alibi_slopes is None and q.dim() == 3:
        _check(lib.fa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, Hq, Hkv, Ncap, d, sc,
                             int(window), _ptr(seqlens_k), hostp, int(num_splits), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(q)))
        return o, lse
    keep, sp = _slopes_ptr(alibi_slopes, Hq, q.device)
    a = DecodeArgs(q=_ptr(q), k=_ptr(k_cache), v=_ptr(v_cache), o=_ptr(o), lse=_ptr(lse), B=B, Hq=Hq, Hkv=Hkv, d=d,
                   scale=sc, window=int(window), Ncap=Ncap, seqlens_k=_ptr(seqlens_k), seqlens_k_host=hostp,
                   num_splits=int(num_splits), workspace=_ptr(workspace),
                   workspace_bytes=workspace.numel() * workspace.element_size(), alibi_slopes=sp, Nq=Nq)
    _check(lib.fa_decode_ex(ctypes.byref(a), _stream(q)))
    return o, lse


def fa_decode_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                    seqlens_k: torch.Tensor, window: int = 0, scale: Optional[float] = None, num_splits: int = 0,
                    seqlens_k_host=None, workspace: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    return_lse: bool = True, alibi_slopes=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Decode over a paged cache: q [B, Hq, d], pages [num_pages, page_size, Hkv, d],
    block_table int32 [B, max_blocks], seqlens_k int32 [B] -> (O [B, Hq, d], LSE [B, Hq]).
    q [B, Nq, Hq, d]: Nq new tokens per sequence, as for fa_decode."""
    lib = load_library()
    _need(q, "q")
    _need(k_pages, "k_pages")
    _need(v_pages, "v_pages")
    _need(block_table, "block_table", torch.int32)
    _need(seqlens_k, "seqlens_k", torch.int32)
    if q.dim() not in (3, 4) or k_pages.dim() != 4 or v_pages.shape != k_pages.shape or block_table.dim() != 2:
        raise FAError(FA_ERR_INVALID, "expected q [B,(Nq,)Hq,d], pages [P,page,Hkv,d], block_table [B,max_blocks]")
    B, Hq, d = q.shape[0], q.shape[-2], q.shape[-1]
    Nq = q.shape[1] if q.dim() == 4 else 1
    num_pages, page_size, Hkv, _ = k_pages.shape
    max_blocks = block_table.shape[1]
    host = _host_ints(seqlens_k_host)
    hostp = _host_ptr(host)
    if workspace is None:
        S = lib.fa_decode_max_splits(B, Hq, Hkv, max_blocks * page_size,
                                     int(window) + Nq - 1 + 63 if window > 0 else 0, hostp, int(num_splits))
        nbytes = lib.fa_decode_workspace_size(B * Nq, Hq, d, max(S, 1))
        workspace = torch.empty((nbytes + 3) // 4, dtype=torch.float32, device=q.device)
    o = out if out is not None else torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Nq) if q.dim() == 4 else (B, Hq), dtype=torch.float32, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    if alibi_slopes is not None or q.dim() == 4:
        keep, sp = _slopes_ptr(alibi_slopes, Hq, q.device)
        a = DecodeArgs(q=_ptr(q), k=_ptr(k_pages), v=_ptr(v_pages), o=_ptr(o), lse=_ptr(lse), B=B, Hq=Hq, Hkv=Hkv,
                       d=d, scale=sc, window=int(window), block_table=_ptr(block_table), max_blocks=max_blocks,
                       page_size=page_size, num_pages=num_pages, seqlens_k=_ptr(seqlens_k), seqlens_k_host=hostp,
                       num_splits=int(num_splits), workspace=_ptr(workspace),
                       workspace_bytes=workspace.numel() * workspace.element_size(), alibi_slopes=sp, Nq=Nq)
        _check(lib.fa_decode_ex(ctypes.byref(a), _stream(q)))
        return o, lse
    _check(lib.fa_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(o), _ptr(lse), B, Hq, Hkv, num_pages,
                               page_size, d, sc, int(window), _ptr(block_table), max_blocks, _ptr(seqlens_k), hostp,
                               int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(q)))
    return o, lse


def fa_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seqlens_k: torch.Tensor,
                      window: int = 0, scale: Optional[float] = None, num_splits: int = 0, seqlens_k_host=None,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      return_lse: bool = True) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """fa_decode whose split partials use the library's fixed per-device scratch (no workspace).

    For callers that cannot allocate device memory; pass ``out``/``lse`` to allocate nothing here
    either.  Calls on one device share the scratch: do not let two of them overlap on the GPU."""
    lib = load_library()
    _need(q, "q")
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache")
    _need(seqlens_k, "seqlens_k", torch.int32)
    B, Hq, d = q.shape
    _, Ncap, Hkv, _ = k_cache.shape
    host = _host_ints(seqlens_k_host)
    o = out if out is not None else torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    _check(lib.fa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, Hq, Hkv, Ncap, d,
                                 sc, int(window), _ptr(seqlens_k), _host_ptr(host),
                                 int(num_splits), _stream(q)))
    return o, lse


def fa_selftest_wait_timeout(limit_ms: int = 20, stream=None) -> None:
    """Launch the library's wait self-test (a wait that nothing completes, limited to limit_ms);
    afterwards fa_device_status() shows the timeout bit (1)."""
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _check(load_library().fa_selftest_wait_timeout(int(limit_ms), ctypes.c_void_p(s)))


def fa_selftest_prefill_abort(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, v_loads: int, causal: bool = False,
                              window: int = 0, alibi_slopes=None, rope=None) -> None:
    """The prefill of fa_fwd on padded q [B, Nq, Hq, d], k/v [B, Nk, Hkv, d] with every CTA's V
    loads cut off after v_loads tiles: the kernel's abort path runs (its waits give up after 2 s)
    and fa_device_status() shows the timeout bit (1).  The outputs are discarded."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    keep, sp = _slopes_ptr(alibi_slopes, Hq, q.device)
    a = FwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), o=_ptr(o), lse=_ptr(lse), B=B, Hq=Hq, Hkv=Hkv, Nq=Nq, Nk=Nk, d=d,
                scale=1.0 / math.sqrt(d), causal=int(bool(causal)), window=int(window), alibi_slopes=sp)
    _set_rope(a, rope, None, d)
    _check(lib.fa_selftest_prefill_abort(ctypes.byref(a), int(v_loads), _stream(q)))
    torch.cuda.synchronize(q.device)  # o, lse and the slopes stay alive until the kernel has ended


def fa_device_status(clear: bool = True) -> int:
    """Synchronise and return the kernels' error bits (0 = clean)."""
    bits = ctypes.c_uint32(0)
    load_library().fa_device_status(ctypes.byref(bits), int(bool(clear)))
    return int(bits.value)
