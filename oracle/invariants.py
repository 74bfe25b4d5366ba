"""Properties every correct result has, checked row by row on the host.

TEST INFRASTRUCTURE ONLY.  For a row with window values v (length L), page
row `pages` (its first ceil(L / page_size) entries) and result `out` (k ints):

  1. count: exactly m = min(k, L) entries are not -1 and they form the prefix;
  2. inverse transform: every entry is page*page_size + o with `page` among the
     row's pages and o < page_size (outputs confined to the row's pages); the
     window indices j it maps back to are distinct, in [0, L) and strictly
     ascending;
  3. threshold: every selected score is >= every unselected score, and where a
     selected and an unselected score are equal, the selected index is lower
     (the tie rule).

The transform is the one of section 1 of the page "[sglang] [AMD ROCm] GLM-5.x
Prefill 성능을 66% 끌어올린 Top-K 커널 최적화 분석".  Inverting it needs the row's
pages to be distinct, which the synthetic page tables guarantee.
"""
from __future__ import annotations

import numpy as np


class InvariantError(AssertionError):
    pass


def check_row(values, pages, page_size: int, k: int, out) -> None:
    """Raises InvariantError when `out` violates one of the properties above."""
    v = np.asarray(values, dtype=np.float32)
    out = np.asarray(out, dtype=np.int64)
    L = int(v.shape[0])
    m = min(k, L)
    if out.shape[0] != k:
        raise InvariantError(f"result has {out.shape[0]} entries, expected k={k}")
    # 1. count and prefix
    if np.any(out[:m] < 0):
        raise InvariantError(f"fewer than min(k, L)={m} entries")
    if np.any(out[m:] != -1):
        raise InvariantError("entries past min(k, L) are not -1")
    if m == 0:
        return
    # 2. inverse transform
    n_pages = (L + page_size - 1) // page_size
    row_pages = np.asarray(pages, dtype=np.int64)[:n_pages]
    if np.unique(row_pages).shape[0] != row_pages.shape[0]:
        raise InvariantError("page row has repeated pages; the transform cannot be inverted")
    page_of = {int(p): idx for idx, p in enumerate(row_pages)}
    sel = out[:m]
    page = sel // page_size
    off = sel % page_size
    try:
        pidx = np.fromiter((page_of[int(p)] for p in page), dtype=np.int64, count=m)
    except KeyError as e:
        raise InvariantError(f"output names page {e} outside the row's pages") from None
    j = pidx * page_size + off
    if np.any(j < 0) or np.any(j >= L):
        raise InvariantError("output maps back outside the window")
    if m > 1 and np.any(np.diff(j) <= 0):
        raise InvariantError("window indices are not strictly ascending")
    # 3. threshold and tie rule
    if m < L:
        mask = np.zeros(L, dtype=bool)
        mask[j] = True
        selected = v[mask]
        unselected = v[~mask]
        lo = selected.min()
        hi = unselected.max()
        if lo < hi:
            raise InvariantError(f"a selected score {lo} is below an unselected one {hi}")
        if lo == hi:
            sel_tied = np.nonzero(mask & (v == lo))[0]
            uns_tied = np.nonzero(~mask & (v == lo))[0]
            if sel_tied.max() > uns_tied.min():
                raise InvariantError("a tie went to a higher window index")


def check_rows(windows, pages_rows, page_size: int, k: int, outs) -> None:
    """check_row over parallel sequences of windows, page rows and results."""
    for r, (w, p, o) in enumerate(zip(windows, pages_rows, outs)):
        try:
            check_row(w, p, page_size, k, o)
        except InvariantError as e:
            raise InvariantError(f"row {r}: {e}") from None
