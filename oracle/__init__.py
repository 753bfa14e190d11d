"""fp64 CPU oracle for paged-KV GQA/MQA attention -- TEST INFRASTRUCTURE.

Loads ``paged_attn_oracle.c`` (compiled with gcc + OpenMP by ``build()``)
through ctypes and marshals numpy arrays into it.  Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package; the CUDA
library and its Python binding never do, and this package never imports them.

What each function computes, and the passages it follows, is written in the
header of ``paged_attn_oracle.c``.  Pins: ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpaged_attn_oracle.so")
_lib = None

F16 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build (portable C, no ISA flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.orc_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64]
    lib.orc_reshape_and_cache.restype = i32
    lib.orc_paged_attention.argtypes = [P, P, P, P, i32, P, P, dbl, i32, i32,
                                        i32, i32, i32, i64, i32, P, i64, P, P,
                                        i32, P, P, i32]
    lib.orc_paged_attention.restype = i32
    lib.orc_cross_attention.argtypes = [P, P, P, P, i32, P, P, dbl, i32, i32,
                                        i32, i32, i32, i64, i32, P, i64, P, P, i32]
    lib.orc_cross_attention.restype = i32
    lib.orc_varlen_attention.argtypes = [P, P, P, P, P, dbl, i32, i32, i32, i32, i32,
                                         P, i64, P, P, i32]
    lib.orc_varlen_attention.restype = i32
    lib.orc_lse_combine.argtypes = [P, P, i64, i32, i32, P]
    lib.orc_lse_combine.restype = None
    lib.orc_to_bits_n.argtypes = [P, i64, i32, P]
    lib.orc_to_bits_n.restype = None
    lib.orc_from_bits_n.argtypes = [P, i64, i32, P]
    lib.orc_from_bits_n.restype = None
    lib.orc_max_threads.argtypes = []
    lib.orc_max_threads.restype = i32
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().orc_max_threads())


def to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round fp64 values to nearest-even fp16/bf16 bit patterns."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_to_bits_n(_ptr(x), x.size, dtype, _ptr(out))
    return out


def from_bits(b: np.ndarray, dtype: int) -> np.ndarray:
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().orc_from_bits_n(_ptr(b), b.size, dtype, _ptr(out))
    return out


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping) -> None:
    """In-place: write k, v [T, Hkv, D] into k_cache, v_cache
    [NB, Hkv, bs, D] at slot_mapping[t] (-1 skips).  Raises on a bad slot."""
    k, v = _c(k, np.uint16), _c(v, np.uint16)
    sm = _c(slot_mapping, np.int64)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    NB, Hkv, bs, D = k_cache.shape
    T = sm.shape[0]
    rc = _load().orc_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache),
                                       _ptr(v_cache), _ptr(sm), T, Hkv, D, bs, NB)
    if rc != 0:
        raise ValueError(f"oracle reshape_and_cache failed: {rc}")


def paged_attention(q, k_cache, v_cache, block_tables, cu_query_lens,
                    context_lens, scale: float, num_kv_heads: int, dtype: int,
                    rows: Optional[np.ndarray] = None, num_splits: int = 1,
                    want_partials: bool = False, num_threads: int = 0):
    """fp64 attention for the query-token rows ``rows`` (default: all).

    Returns (out64 [n, Hq, D], out_bits [n, Hq, D] uint16) and, with
    ``want_partials`` and num_splits > 1, also (part_o [n, Hq, S, D],
    part_lse [n, Hq, S]).
    """
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_query_lens, np.int32)
    ctx = _c(context_lens, np.int32)
    Tq, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and Hkv == num_kv_heads
    B = ctx.shape[0]
    mbs = bt.shape[1] if bt.ndim == 2 else 0
    rows_a = None if rows is None else _c(rows, np.int64)
    n = Tq if rows_a is None else rows_a.shape[0]
    out64 = np.zeros((n, Hq, D), np.float64)
    outb = np.zeros((n, Hq, D), np.uint16)
    S = max(1, int(num_splits))
    po = pl = None
    if want_partials and S > 1:
        po = np.zeros((n, Hq, S, D), np.float64)
        pl = np.zeros((n, Hq, S), np.float64)
    rc = _load().orc_paged_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), mbs, _ptr(cu),
        _ptr(ctx), float(scale), B, Hq, Hkv, D, bs, NB, dtype, _ptr(rows_a),
        n, _ptr(out64), _ptr(outb), S, _ptr(po), _ptr(pl), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle paged_attention failed: {rc}")
    if want_partials and S > 1:
        return out64, outb, po, pl
    return out64, outb


def cross_attention(q, k_cache, v_cache, block_tables, cu_query_lens,
                    context_lens, scale: float, num_kv_heads: int, dtype: int,
                    rows: Optional[np.ndarray] = None, num_threads: int = 0):
    """fp64 cross-attention (no causal mask: every query row of a sequence
    sees all of its context_lens cached keys) for the query-token rows
    ``rows`` (default: all).  Returns (out64 [n, Hq, D], out_bits)."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_query_lens, np.int32)
    ctx = _c(context_lens, np.int32)
    Tq, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and Hkv == num_kv_heads
    B = ctx.shape[0]
    mbs = bt.shape[1] if bt.ndim == 2 else 0
    rows_a = None if rows is None else _c(rows, np.int64)
    n = Tq if rows_a is None else rows_a.shape[0]
    out64 = np.zeros((n, Hq, D), np.float64)
    outb = np.zeros((n, Hq, D), np.uint16)
    rc = _load().orc_cross_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), mbs, _ptr(cu),
        _ptr(ctx), float(scale), B, Hq, Hkv, D, bs, NB, dtype, _ptr(rows_a),
        n, _ptr(out64), _ptr(outb), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle cross_attention failed: {rc}")
    return out64, outb


def varlen_attention(q, k, v, cu_q, cu_k, scale: float, dtype: int,
                     rows: Optional[np.ndarray] = None, num_threads: int = 0):
    """fp64 GQA prefill over contiguous K/V of a varlen batch: q [Tq, Hq, D],
    k, v [Tk, Hkv, D], bottom-right causal per sequence.  Returns
    (out64 [n, Hq, D], out_bits)."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    cq, ck = _c(cu_q, np.int32), _c(cu_k, np.int32)
    Tq, Hq, D = q.shape
    Tk, Hkv, D2 = k.shape
    assert D2 == D and v.shape == k.shape and cq.shape == ck.shape
    B = cq.shape[0] - 1
    rows_a = None if rows is None else _c(rows, np.int64)
    n = Tq if rows_a is None else rows_a.shape[0]
    out64 = np.zeros((n, Hq, D), np.float64)
    outb = np.zeros((n, Hq, D), np.uint16)
    rc = _load().orc_varlen_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck),
                                      float(scale), B, Hq, Hkv, D, dtype, _ptr(rows_a), n,
                                      _ptr(out64), _ptr(outb), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle varlen_attention failed: {rc}")
    return out64, outb


def lse_combine(part_o: np.ndarray, part_lse: np.ndarray) -> np.ndarray:
    """Combine split partials: part_o [..., S, D], part_lse [..., S]."""
    po = _c(part_o, np.float64)
    pl = _c(part_lse, np.float64)
    S, D = po.shape[-2], po.shape[-1]
    n = int(np.prod(po.shape[:-2]))
    out = np.zeros(po.shape[:-2] + (D,), np.float64)
    _load().orc_lse_combine(_ptr(po), _ptr(pl), n, S, D, _ptr(out))
    return out


def run_case(case, rows: Optional[np.ndarray] = None, num_threads: int = 0):
    """The whole step of a workload case on the CPU: reshape_and_cache of the
    case's new tokens into a copy of its cache, then attention for ``rows``.
    Returns (out64, out_bits, k_cache_after, v_cache_after)."""
    kc = case.k_cache.copy()
    vc = case.v_cache.copy()
    if getattr(case, "cross", False):  # static encoder cache: nothing to write
        o64, ob = cross_attention(case.q, kc, vc, case.block_tables,
                                  case.cu_query_lens, case.context_lens, case.scale,
                                  case.num_kv_heads, case.dtype, rows=rows,
                                  num_threads=num_threads)
        return o64, ob, kc, vc
    reshape_and_cache(case.k_new, case.v_new, kc, vc, case.slot_mapping)
    o64, ob = paged_attention(case.q, kc, vc, case.block_tables,
                              case.cu_query_lens, case.context_lens, case.scale,
                              case.num_kv_heads, case.dtype, rows=rows,
                              num_threads=num_threads)
    return o64, ob, kc, vc
