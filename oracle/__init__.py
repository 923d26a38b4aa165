"""CPU oracle for the paged-attention decode read (TEST INFRASTRUCTURE).

This package is the correctness reference the CUDA library is graded
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may import it; the product package never does, and the two
share no code.

The arithmetic lives in ``np_oracle.c`` / ``decode_body.h`` (plain C loops,
gathered history + exact two-pass softmax, see the header comment there for
the passages each step follows).  This module only marshals numpy arrays into
that library with ctypes.

Array conventions (numpy, C-contiguous):
  * fp32 data is ``np.float32``; bf16 data is its raw bit pattern as
    ``np.uint16`` (numpy has no bf16 type).
  * q [rows, q_heads, head_dim]; pools [num_blocks, block_size, kv_heads,
    head_dim]; block_tables [rows, max_blocks_per_row] int32; context_lens
    [rows] int32; slot_mapping [num_tokens] int64.
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np

from . import build as _build

F32 = 0
BF16 = 1

OK = 0
BAD_ARG = 1
BAD_BLOCK = 2
BAD_CONTEXT = 3
NO_MEMORY = 4

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_LIB = None
_LOAD_LOCK = threading.Lock()


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} returned {code}")
        self.code = code


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _LIB
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _LOAD_LOCK:  # host threads may call the oracle at once
        if _LIB is None:
            _LIB = _declare(ctypes.CDLL(_build.build()))
    return _LIB


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.npo_widen.restype = ctypes.c_double
    lib.npo_widen.argtypes = [_P, ctypes.c_int, _I64]
    lib.npo_kv_append.restype = ctypes.c_int
    lib.npo_kv_append.argtypes = [_P, _P, ctypes.c_int, _I64, _I32, _I32, _I32,
                                  _P, _P, _P, _I32]
    for name in ("npo_paged_decode_f64", "npo_paged_decode_f32"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [_P, _P, _P, _P, _P, ctypes.c_int, _I64, _I32, _I32, _I32,
                       _P, _I32, _P, _I32, _I32, _I32, ctypes.c_double, _I64, _I32]
    lib.npo_reduce_f64.restype = ctypes.c_int
    lib.npo_reduce_f64.argtypes = [_P, _P, _P, _I32, _I32, _I32, _I32]
    return lib


def dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or bf16 bits (uint16), got {a.dtype}")


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype=None) -> np.ndarray:
    return np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))


def paged_decode(q, k_pool, v_pool, block_tables, context_lens, scale, *,
                 split_len: int | None = None, num_splits: int = 1,
                 precision: str = "f64", lib: ctypes.CDLL | None = None):
    """Decode read over the paged pool.

    ``q`` is [rows, q_heads, head_dim] (one query token per row) or
    [rows, query_len, q_heads, head_dim] (query token i of row r sits at
    position context_lens[r] - query_len + i and sees the history up to it).
    Returns ``(out, lse)`` with q's leading shape: out [..., q_heads,
    head_dim] and lse [..., q_heads] when ``num_splits == 1``; otherwise the
    per-split partials out [..., q_heads, num_splits, head_dim] and lse
    [..., q_heads, num_splits], split s covering tokens
    [s * split_len, (s + 1) * split_len).  ``precision`` is "f64" (the primary
    oracle) or "f32".
    """
    lib = lib or load()
    q, k_pool, v_pool = _c(q), _c(k_pool), _c(v_pool)
    code = dtype_code(q)
    if dtype_code(k_pool) != code or dtype_code(v_pool) != code:
        raise TypeError("q and both pools must share one dtype")
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    multi = q.ndim == 4
    if multi:
        rows, query_len, q_heads, head_dim = q.shape
    else:
        rows, q_heads, head_dim = q.shape
        query_len = 1
    num_blocks, block_size, kv_heads, hd2 = k_pool.shape
    if hd2 != head_dim or v_pool.shape != k_pool.shape:
        raise ValueError("pool shape does not match q")
    if bt.ndim != 2 or bt.shape[0] != rows:
        raise ValueError("block_tables must be [rows, max_blocks_per_row]")
    mb = bt.shape[1]
    if split_len is None:
        split_len = max(1, mb * block_size)
    real = np.float64 if precision == "f64" else np.float32
    fn = lib.npo_paged_decode_f64 if precision == "f64" else lib.npo_paged_decode_f32
    out = np.zeros((rows, query_len, q_heads, num_splits, head_dim), dtype=real)
    lse = np.zeros((rows, query_len, q_heads, num_splits), dtype=real)
    rc = fn(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_pool), _ptr(v_pool), code,
            num_blocks, block_size, kv_heads, head_dim, _ptr(bt), mb, _ptr(cl),
            rows, query_len, q_heads, float(scale), int(split_len), num_splits)
    if rc != OK:
        raise OracleError(rc, "paged_decode")
    if not multi:
        out, lse = out[:, 0], lse[:, 0]
    if num_splits == 1:
        return out[..., 0, :], lse[..., 0]
    return out, lse


def kv_append(k_pool, v_pool, k_new, v_new, slot_mapping, *, lib=None) -> int:
    """Scatter the new tokens' K/V rows into the pools IN PLACE.

    Returns the oracle status: OK, or BAD_BLOCK if some slot lies past the
    pool (those tokens are skipped; negative slots are skipped silently).
    """
    lib = lib or load()
    for a in (k_pool, v_pool):
        if not a.flags.c_contiguous:
            raise ValueError("pools must be C-contiguous (written in place)")
    num_blocks, block_size, kv_heads, head_dim = k_pool.shape
    # [R, Q, Hk, D] tokens with [R, Q] slots are R*Q tokens
    k_new = _c(k_new).reshape(-1, kv_heads, head_dim)
    v_new = _c(v_new).reshape(-1, kv_heads, head_dim)
    code = dtype_code(k_pool)
    sm = _c(slot_mapping, np.int64).reshape(-1)
    n = sm.shape[0]
    if k_new.shape != (n, kv_heads, head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens, kv_heads, head_dim]")
    return lib.npo_kv_append(_ptr(k_pool), _ptr(v_pool), code, num_blocks,
                             block_size, kv_heads, head_dim, _ptr(k_new),
                             _ptr(v_new), _ptr(sm), n)


def reduce(o_part, lse_part, *, lib=None) -> np.ndarray:
    """Log-sum-exp combine of split partials (fp64): [R,Hq,S,D],[R,Hq,S] -> [R,Hq,D]."""
    lib = lib or load()
    o = _c(o_part, np.float64)
    lse = _c(lse_part, np.float64)
    rows, q_heads, num_splits, head_dim = o.shape
    out = np.zeros((rows, q_heads, head_dim), dtype=np.float64)
    rc = lib.npo_reduce_f64(_ptr(out), _ptr(o), _ptr(lse), rows, q_heads,
                            num_splits, head_dim)
    if rc != OK:
        raise OracleError(rc, "reduce")
    return out


def widen(a: np.ndarray, idx: int, *, lib=None) -> float:
    """The oracle's own widening of element ``idx`` of ``a`` to double."""
    lib = lib or load()
    a = _c(a)
    return lib.npo_widen(_ptr(a), dtype_code(a), int(idx))
