"""fp64 CPU oracle for exact attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  It shares no code with the CUDA library ``exact_io_aware_09_gb300``
and never imports it.

Contents
  * ``attn_oracle.c`` (built to ``liboracle.so``): the three-step materialising definition of
    attention in fp64, the FA-2 online recurrence and the (m, l, o) merge for the pages'
    worked traces, and exact fp16/bf16 conversions.
  * ``bytes_model.py``: the logical HBM-traffic model of "FlashAttention and GPU Data
    Movement", sections 1.1 and 4.
  * ``tiles.py``: the causal skip bound and diagonal-mask tile listing of the same page,
    section 2.1 and exercise 4.

Parity status of each function is stated in its docstring; every function here is pinned
by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .bytes_model import bytes_model, flash_traffic, naive_traffic  # noqa: F401
from .tiles import causal_tiles  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# A prebuilt copy of the library to load instead (the mutation check of the pins builds copies
# of attn_oracle.c with one planted mistake each and runs the pins against them).
_LIB_OVERRIDE = os.environ.get("ORACLE_LIB_OVERRIDE")
_lock = threading.Lock()
_lib = None
_tables = {}

F16, BF16 = 0, 1
_DT = {"f16": F16, "bf16": BF16, F16: F16, BF16: BF16}


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (plain -O2, IEEE semantics, OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if _LIB_OVERRIDE:
            lib = ctypes.CDLL(_LIB_OVERRIDE)
        else:
            build()
            lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_attention_rows.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                              f64, P, i64, P, P, i32]
        lib.oracle_attention_rows.restype = i32
        lib.oracle_attention_rows_masked.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                     i32, i64, P, i32, f64, P, i64, P, P, i32]
        lib.oracle_attention_rows_masked.restype = i32
        lib.oracle_round_to_storage.argtypes = [P, P, i64, i32]
        lib.oracle_round_to_storage.restype = None
        lib.oracle_decode_rows.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f64, P, i64,
                                           P, P, i32]
        lib.oracle_decode_rows.restype = i32
        lib.oracle_online_trace.argtypes = [P, P, i32, i32, P, i32, P, P, P, P, P]
        lib.oracle_online_trace.restype = i32
        lib.oracle_merge_states.argtypes = [f64, f64, P, f64, f64, P, i32, P, P, P]
        lib.oracle_merge_states.restype = None
        lib.oracle_block_summary.argtypes = [P, i32, P, P]
        lib.oracle_block_summary.restype = None
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = f64
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = f64
        lib.oracle_double_to_f16.argtypes = [f64]
        lib.oracle_double_to_f16.restype = ctypes.c_uint16
        lib.oracle_double_to_bf16.argtypes = [f64]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


# ----------------------------------------------------------------------------------------
# conversions
# ----------------------------------------------------------------------------------------
def f16_to_double(bits: int) -> float:
    return float(_load().oracle_f16_to_double(int(bits) & 0xFFFF))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits) & 0xFFFF))


def double_to_f16(x: float) -> int:
    """Round to the nearest binary16, ties to even; returns the bit pattern."""
    return int(_load().oracle_double_to_f16(float(x)))


def double_to_bf16(x: float) -> int:
    return int(_load().oracle_double_to_bf16(float(x)))


def round_to_storage(x: np.ndarray, dtype) -> np.ndarray:
    """Storage bits of x rounded to fp16 / bf16 (nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_to_storage(_ptr(x), _ptr(out), x.size, _DT[dtype])
    return out


def bits_to_double(bits: np.ndarray, dtype) -> np.ndarray:
    """Exact fp64 values of an array of fp16/bf16 bit patterns (via the oracle's table)."""
    key = _DT[dtype]
    table = _tables.get(key)
    if table is None:
        lib = _load()
        conv = lib.oracle_bf16_to_double if key == BF16 else lib.oracle_f16_to_double
        table = np.array([conv(i) for i in range(65536)], dtype=np.float64)
        _tables[key] = table
    return table[np.asarray(bits, dtype=np.uint16)]


# ----------------------------------------------------------------------------------------
# the definition
# ----------------------------------------------------------------------------------------
def attention_rows(q, k, v, dtype, B, Hq, Hkv, Nq, Nkv, d, causal, scale, rows=None,
                   threads: int = 0, window=None, block_mask=None, block: int = 128):
    """O and L of the materialising definition for selected query rows.

    q, k, v: uint16 bit arrays, shapes [B,Hq,Nq,d] and [B,Hkv,Nkv,d].
    rows: flat indices (b*Hq + h)*Nq + i; ``None`` = every row.
    window: sliding window W (key j visible to row i iff 0 <= i + Nkv - Nq - j <= W), or None.
    block_mask: [ceil(Nq/block), ceil(Nkv/block)] pattern of blocks to compute, or None.
    Returns (o [n_rows, d] float64, lse [n_rows] float64).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    assert q.size == B * Hq * Nq * d and k.size == B * Hkv * Nkv * d and v.size == k.size
    if rows is None:
        rows = np.arange(B * Hq * Nq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.zeros((len(rows), d), dtype=np.float64)
    lse = np.zeros(len(rows), dtype=np.float64)
    if block_mask is not None:
        block_mask = np.ascontiguousarray(block_mask, dtype=np.uint8)
        assert block_mask.shape == (-(-Nq // block), -(-Nkv // block)), block_mask.shape
    rc = _load().oracle_attention_rows_masked(
        _ptr(q), _ptr(k), _ptr(v), _DT[dtype], B, Hq, Hkv, Nq, Nkv, d, int(bool(causal)),
        -1 if window is None else int(window),
        _ptr(block_mask) if block_mask is not None else None, int(block), float(scale),
        _ptr(rows), len(rows), _ptr(o), _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle_attention_rows: bad arguments")
    return o, lse


def attention(q, k, v, dtype, B, Hq, Hkv, Nq, Nkv, d, causal, scale, threads: int = 0):
    o, lse = attention_rows(q, k, v, dtype, B, Hq, Hkv, Nq, Nkv, d, causal, scale, None,
                            threads)
    return o.reshape(B, Hq, Nq, d), lse.reshape(B, Hq, Nq)


def gather_pages(pages, block_table, seqlens, page_size):
    """The packed [sum(L), Hkv, d] cache of a paged one: sequence b's token t is row
    t % page_size of page block_table[b][t // page_size] ("FlashAttention Explained", section
    "Decoding, Paged and Split-KV Variants": fixed-size non-contiguous blocks addressed through
    a block table).  pages: [num_pages, page_size, Hkv, d]."""
    pages = np.asarray(pages)
    out = []
    for b, L in enumerate(np.asarray(seqlens, dtype=np.int64)):
        t = np.arange(int(L), dtype=np.int64)
        out.append(pages[np.asarray(block_table)[b][t // page_size], t % page_size])
    if not out:
        return pages[:0, 0]
    return np.ascontiguousarray(np.concatenate(out, axis=0))


def decode_rows_paged(q, k_pages, v_pages, block_table, seqlens, page_size, dtype, B, Hq, Hkv,
                      d, scale, rows=None, threads: int = 0):
    """Decode attention over a paged cache: the packed definition of the gathered cache."""
    seqlens = np.asarray(seqlens, dtype=np.int64)
    kc = gather_pages(k_pages, block_table, seqlens, page_size)
    vc = gather_pages(v_pages, block_table, seqlens, page_size)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    return decode_rows(q, kc, vc, cu, dtype, B, Hq, Hkv, d, scale, rows, threads)


def decode_rows(q, k_cache, v_cache, cu_seqlens, dtype, B, Hq, Hkv, d, scale, rows=None,
                threads: int = 0):
    """Decode attention (one query token per sequence, packed [T, Hkv, d] cache).

    rows: flat indices b*Hq + h; ``None`` = all.  Returns (o [n_rows, d], lse [n_rows]).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint16)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint16)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    assert q.size == B * Hq * d and len(cu) == B + 1 and kc.size == int(cu[-1]) * Hkv * d
    if rows is None:
        rows = np.arange(B * Hq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.zeros((len(rows), d), dtype=np.float64)
    lse = np.zeros(len(rows), dtype=np.float64)
    rc = _load().oracle_decode_rows(_ptr(q), _ptr(kc), _ptr(vc), _ptr(cu), _DT[dtype], B, Hq,
                                    Hkv, d, float(scale), _ptr(rows), len(rows), _ptr(o),
                                    _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle_decode_rows: bad arguments")
    return o, lse


# ----------------------------------------------------------------------------------------
# the method's steps (for the pages' worked traces)
# ----------------------------------------------------------------------------------------
def online_trace(scores, values, block_ends):
    """FA-2 online recurrence over blocks of one row.

    Returns dict with per-block m, l, alpha, a (after the block) and the final o = a / l.
    """
    s = np.ascontiguousarray(scores, dtype=np.float64)
    vals = np.asarray(values, dtype=np.float64)
    if vals.ndim == 1:
        vals = vals[:, None]
    vals = np.ascontiguousarray(vals)
    n, dv = vals.shape
    assert len(s) == n
    ends = np.ascontiguousarray(block_ends, dtype=np.int32)
    nb = len(ends)
    m = np.zeros(nb)
    l = np.zeros(nb)
    al = np.zeros(nb)
    a = np.zeros((nb, dv))
    o = np.zeros(dv)
    rc = _load().oracle_online_trace(_ptr(s), _ptr(vals), n, dv, _ptr(ends), nb, _ptr(m),
                                     _ptr(l), _ptr(al), _ptr(a), _ptr(o))
    if rc != 0:
        raise ValueError("oracle_online_trace: bad block ends")
    return {"m": m, "l": l, "alpha": al, "a": a, "o": o}


def merge_states(s1, s2):
    """Merge two (m, l, o) states, o normalised within its block."""
    m1, l1, o1 = s1
    m2, l2, o2 = s2
    o1 = np.ascontiguousarray(np.atleast_1d(o1), dtype=np.float64)
    o2 = np.ascontiguousarray(np.atleast_1d(o2), dtype=np.float64)
    dv = len(o1)
    m = np.zeros(1)
    l = np.zeros(1)
    o = np.zeros(dv)
    _load().oracle_merge_states(float(m1), float(l1), _ptr(o1), float(m2), float(l2), _ptr(o2),
                                dv, _ptr(m), _ptr(l), _ptr(o))
    return float(m[0]), float(l[0]), o


def block_summary(x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    m = np.zeros(1)
    l = np.zeros(1)
    _load().oracle_block_summary(_ptr(x), len(x), _ptr(m), _ptr(l))
    return float(m[0]), float(l[0])
