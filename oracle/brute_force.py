"""Selection by closed-form rank, in pure Python, for tiny rows.

TEST INFRASTRUCTURE ONLY.  An implementation of the selection rule that uses
no sort at all, so that it pins the C oracle independently:

    rank_j = #{a : v_a > v_j} + #{a < j : v_a == v_j}

is the position of element j in the order (score descending, index
ascending); element j is selected iff rank_j < k.  Selected indices are then
listed in ascending order, mapped through the page transform of section 1 of
the page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66% 끌어올린 Top-K 커널
최적화 분석" (page_row[j >> page_bits] * page_size + (j & (page_size-1))),
and padded with -1 to k.  Python float comparison treats -0.0 == +0.0.
"""
from __future__ import annotations


def select_by_rank(values, k: int) -> list[int]:
    """Window indices with rank < k, ascending."""
    n = len(values)
    chosen = []
    for j in range(n):
        vj = values[j]
        rank = 0
        for a in range(n):
            va = values[a]
            if va > vj or (a < j and va == vj):
                rank += 1
        if rank < k:
            chosen.append(j)
    return chosen


def select_by_rank_np(values, k: int):
    """The same closed-form rank, evaluated for all j at once with numpy
    broadcasting (O(n^2) memory: tiny rows only).  Returns ascending indices."""
    import numpy as np

    v = np.asarray(values, dtype=np.float64)
    n = v.shape[0]
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    greater = (v[None, :] > v[:, None]).sum(axis=1)
    idx = np.arange(n)
    earlier_equal = ((v[None, :] == v[:, None]) & (idx[None, :] < idx[:, None])).sum(axis=1)
    rank = greater + earlier_equal
    return np.nonzero(rank < k)[0]


def page_slot(page_row, page_size: int, j: int) -> int:
    """Section 1's transform with page_bits = log2(page_size): the page from
    the high bits of j, the offset inside the page from the low bits."""
    page_bits = page_size.bit_length() - 1
    return int(page_row[j >> page_bits]) * page_size + (j & (page_size - 1))


def row_result(values, page_row, page_size: int, k: int) -> list[int]:
    """page_row None: raw window indices (the identity transform)."""
    chosen = select_by_rank(values, k)
    out = list(chosen) if page_row is None else [page_slot(page_row, page_size, j) for j in chosen]
    return out + [-1] * (k - len(out))


def packed_result(scores_flat, row_stride: int, seq_lens, row_starts, row_to_batch,
                  page_table_flat, pt_stride: int, page_size: int, k: int) -> list[list[int]]:
    """All rows of a packed problem (plain Python lists/sequences)."""
    rows = []
    for i in range(len(seq_lens)):
        n = max(int(seq_lens[i]), 0)
        base = i * row_stride + int(row_starts[i])
        values = [float(scores_flat[base + j]) for j in range(n)]
        b = i if row_to_batch is None else int(row_to_batch[i])
        if page_table_flat is None:
            page_row = None
        else:
            pages_needed = (n + page_size - 1) // page_size
            page_row = [int(page_table_flat[b * pt_stride + p]) for p in range(pages_needed)]
        rows.append(row_result(values, page_row, page_size, k))
    return rows
