"""ctypes wrappers over the C oracle (oracle.c).  Test infrastructure only.

All arrays are numpy; 16-bit token data is passed as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None
_P = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_slot_mapping.argtypes = [_P, _P, ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int]
        L.oracle_slot_mapping.restype = None
        L.oracle_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P] + [ctypes.c_int] * 4 + [_P]
        L.oracle_reshape_and_cache.restype = None
        L.oracle_copy_blocks.argtypes = [_P, _P, _P] + [ctypes.c_int] * 4 + [_P]
        L.oracle_copy_blocks.restype = None
        L.oracle_swap_blocks.argtypes = [_P] * 5 + [ctypes.c_int] * 4
        L.oracle_swap_blocks.restype = None
        L.oracle_decode.argtypes = ([_P] * 6 + [ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_int]
                                    + [_P, _P, ctypes.c_int, ctypes.c_int])
        L.oracle_decode.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def f16_to_double(bits: int) -> float:
    return lib().oracle_f16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def slot_mapping(block_tables, seq_idx, pos, block_size) -> np.ndarray:
    bt = _c(block_tables, np.int32)
    si, ps = _c(seq_idx, np.int32), _c(pos, np.int32)
    T = len(si)
    out = np.empty(T, dtype=np.int64)
    lib().oracle_slot_mapping(_ptr(out), _ptr(bt), bt.shape[1], _ptr(si), _ptr(ps), T, block_size)
    return out


def reshape_and_cache(k_cache, v_cache, key, value, slots, row_of_block=None):
    """In place on k_cache/v_cache ([rows, bs, H, D] uint16, C-contiguous)."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    _, bs, H, D = k_cache.shape
    key, value = _c(key, np.uint16), _c(value, np.uint16)
    sl = _c(slots, np.int64)
    rob = _c(row_of_block, np.int32)
    lib().oracle_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), _ptr(key), _ptr(value), _ptr(sl),
                                   len(sl), H, D, bs, _ptr(rob))


def copy_blocks(k_cache, v_cache, pairs, row_of_block=None):
    """In place; pairs: [P, 2] (src, dst) physical block ids."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    _, bs, H, D = k_cache.shape
    pr = _c(np.asarray(pairs, dtype=np.int64).reshape(-1, 2), np.int64)
    rob = _c(row_of_block, np.int32)
    lib().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pr), pr.shape[0], H, D, bs,
                             _ptr(rob))


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs):
    """In place on dst_k/dst_v; pairs: [P, 2] (src block, dst block)."""
    for a in (dst_k, dst_v, src_k, src_v):
        assert a.flags.c_contiguous and a.dtype == np.uint16
    _, bs, H, D = src_k.shape
    pr = _c(np.asarray(pairs, dtype=np.int64).reshape(-1, 2), np.int64)
    lib().oracle_swap_blocks(_ptr(dst_k), _ptr(dst_v), _ptr(src_k), _ptr(src_v), _ptr(pr),
                             pr.shape[0], H, D, bs)


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, is_bf16,
           row_of_block=None, items=None, nthreads=1) -> np.ndarray:
    """fp64 decode attention; returns out [S, H, D] float64.

    items: optional [n, 2] (seq, head) pairs to compute; others stay NaN.
    """
    q = _c(q, np.uint16)
    S, H, D = q.shape
    bs = k_cache.shape[1]
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    rob = _c(row_of_block, np.int32)
    it = None if items is None else _c(np.asarray(items).reshape(-1, 2), np.int32)
    out = np.full((S, H, D), np.nan, dtype=np.float64)
    rc = lib().oracle_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl),
                             S, H, D, bs, bt.shape[1], float(scale), int(bool(is_bf16)), _ptr(rob),
                             _ptr(it), 0 if it is None else it.shape[0], int(nthreads))
    assert rc == 0
    return out


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)
