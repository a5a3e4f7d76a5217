"""fp64 CPU oracle for the attention forward — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and ``bench.py --impl reference``) may import anything in this package.
The product path (the CUDA library and its Python binding) never does, and the
oracle never imports the product.

Two independent implementations:

* ``attention_ref.c`` (``attention_rows``): plain C, one output row at a time,
  OpenMP over rows; used for parity at every size, including sampled rows of
  the largest workloads, and for the timed CPU baseline.
* ``ref_numpy`` (``attention``, ``merge_partials``): numpy, whole score matrix
  per (sequence, head); used to cross-check the C oracle on small inputs.

Parity status: pinned.  ``tests/test_oracle.py`` checks both against
brute-force loops, ``torch.nn.functional.scaled_dot_product_attention`` in
float64 on the CPU (a library special case), closed forms and invariants.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .ref_numpy import attention as attention_numpy  # noqa: F401
from .ref_numpy import merge_partials, visible_mask  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_ref.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attention_ref.c`` into ``liboracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention_rows(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray,
                   q_off, len_q, k_off, len_k, scale: float, causal: bool, window: int,
                   rows: np.ndarray, threads: int = 0, alibi_slopes=None):
    """Selected rows of attention, in fp64, from bf16 bit patterns.

    q_bits [Tq, Hq, d] uint16, k_bits/v_bits [Tk, Hkv, d] uint16 (row-major).
    Sequence b occupies q rows q_off[b] .. q_off[b]+len_q[b]-1 (same for k).
    rows: int array [n, 3] of (b, h, i).  Returns (O [n, d], LSE [n]) float64.
    alibi_slopes: optional per-query-head slopes m_h; the score gets -m_h |p - j|.
    """
    lib = _load()
    # leading dims are flattened into rows: [..., H, d] -> [rows, H, d]
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    q_bits = q_bits.reshape(-1, q_bits.shape[-2], q_bits.shape[-1])
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    k_bits = k_bits.reshape(-1, k_bits.shape[-2], k_bits.shape[-1])
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    v_bits = v_bits.reshape(-1, v_bits.shape[-2], v_bits.shape[-1])
    _, hq, d = q_bits.shape
    hkv = k_bits.shape[1]
    B = len(len_q)
    q_off = np.ascontiguousarray(q_off, dtype=np.int64)
    k_off = np.ascontiguousarray(k_off, dtype=np.int64)
    len_q = np.ascontiguousarray(len_q, dtype=np.int32)
    len_k = np.ascontiguousarray(len_k, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    n = rows.shape[0]
    slopes = None if alibi_slopes is None else np.ascontiguousarray(alibi_slopes, dtype=np.float64)
    if slopes is not None and slopes.shape != (hq,):
        raise ValueError("alibi_slopes must have one slope per query head")
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_attention_rows(
        _ptr(q_bits), _ptr(k_bits), _ptr(v_bits),
        ctypes.c_int(B), ctypes.c_int(hq), ctypes.c_int(hkv), ctypes.c_int(d),
        _ptr(q_off), _ptr(len_q), _ptr(k_off), _ptr(len_k),
        ctypes.c_double(scale), ctypes.c_int(int(bool(causal))), ctypes.c_int(int(window)),
        _ptr(slopes) if slopes is not None else None,
        ctypes.c_int(n), _ptr(rows), _ptr(o), _ptr(lse), ctypes.c_int(int(threads)))
    if rc != 0:
        raise ValueError("oracle_attention_rows: bad arguments or out of memory")
    return o, lse


def all_rows(len_q, hq: int) -> np.ndarray:
    """Every (b, h, i) triple, ordered b, h, i."""
    out = []
    for b, lq in enumerate(len_q):
        for h in range(hq):
            if lq > 0:
                blk = np.empty((lq, 3), dtype=np.int32)
                blk[:, 0] = b
                blk[:, 1] = h
                blk[:, 2] = np.arange(lq)
                out.append(blk)
    return np.concatenate(out) if out else np.zeros((0, 3), dtype=np.int32)
