"""CPU oracle for the packed-layout top-k + page transform.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it.  The library (``sparse_attention_top_packed_b300``)
never imports it, and it imports nothing from the library.

Contents
  * :func:`topk_packed_reference` -- the definition computed by the C oracle
    (``topk_oracle.c``): per row, a full sort by (score descending, index
    ascending), the first min(k, seq_len) indices in ascending order, the page
    transform, -1 padding.
  * :mod:`oracle.brute_force` -- the same selection from the closed-form rank of
    each element, in pure Python, for tiny rows (pins the C oracle).
  * :mod:`oracle.invariants` -- properties every correct output has.

Source of the operation: page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66%
끌어올린 Top-K 커널 최적화 분석" (analysis of sglang PR #37889), Intro (packed
layout), section 1 "TopKPackedParams" (window, table row, page transform) and
section 2 (masked lanes never win).  The page leaves the selection rule, the
output order, the tie rule and the padding unstated; the rule implemented is
the library's specification: k largest, ties to the lower window index,
ascending window index, -1 padding.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        if not _build.up_to_date():
            _build.build()
        lib = ctypes.CDLL(_build.LIBRARY)
        lib.topk_oracle.restype = ctypes.c_int
        lib.topk_oracle.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
            ctypes.c_int32, ctypes.c_int32,
        ]
        lib.topk_oracle_typed.restype = ctypes.c_int
        lib.topk_oracle_typed.argtypes = [
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
            ctypes.c_int32, ctypes.c_int32,
        ]
        lib.topk_oracle_default_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    """Threads the C oracle uses when not told otherwise (one per online core)."""
    return int(_load().topk_oracle_default_threads())


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


DTYPES = {"f32": 0, "bf16": 1, "f16": 2}


def topk_packed_reference(scores, row_stride: int, seq_lens, row_starts, row_to_batch,
                          page_table, pt_stride: int, page_size: int, k: int,
                          num_rows: int | None = None, nthreads: int = 0, dtype: str = "f32") -> np.ndarray:
    """Returns the [num_rows, k] int32 result of the definition for host arrays.

    ``scores`` is read at ``i*row_stride + row_starts[i] + j``: a float32
    array (dtype "f32"), or the 16-bit patterns of bfloat16 ("bf16") or IEEE
    binary16 ("f16") values as a uint16 (or float16) array;
    ``row_to_batch`` may be None (identity); ``page_table`` is read at
    ``b*pt_stride + page``, or is None for raw window indices (no page
    transform).  ``nthreads <= 0`` uses every online core.
    """
    lib = _load()
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    if dtype == "f32":
        sc = np.ascontiguousarray(np.asarray(scores, dtype=np.float32)).reshape(-1)
    else:
        a = np.asarray(scores)
        if a.dtype not in (np.uint16, np.int16, np.float16):
            raise ValueError("16-bit scores must be given as their bit patterns (uint16) or float16")
        sc = np.ascontiguousarray(a.view(np.uint16)).reshape(-1)
    sl = _i32(seq_lens)
    rs = _i32(row_starts)
    rb = None if row_to_batch is None else _i32(row_to_batch)
    pt = None if page_table is None else _i32(page_table).reshape(-1)
    n = int(sl.shape[0]) if num_rows is None else int(num_rows)
    if sl.shape[0] < n or rs.shape[0] < n or (rb is not None and rb.shape[0] < n):
        raise ValueError("per-row arrays are shorter than num_rows")
    if k <= 0:
        raise ValueError("k must be positive")
    out = np.empty((n, k), dtype=np.int32)
    if pt is not None and pt.size == 0:
        pt = np.zeros(1, dtype=np.int32)
    rc = lib.topk_oracle_typed(sc.ctypes.data, DTYPES[dtype], int(row_stride), sl.ctypes.data, rs.ctypes.data,
                         None if rb is None else rb.ctypes.data, None if pt is None else pt.ctypes.data,
                         int(pt_stride),
                         int(page_size), int(k), out.ctypes.data, n, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return out


__all__ = ["topk_packed_reference", "default_threads"]
