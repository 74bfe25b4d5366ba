"""Test helpers for GPU parity: copy windows to the host for the CPU oracle,
and check the result's invariants on every row with torch ops on the device.
Nothing here computes an expected result: expected values come from the oracle."""
from __future__ import annotations

import numpy as np
import torch

from oracle import topk_packed_reference
from sparse_attention_top_packed_b300.workloads import gather_windows, sample_rows  # noqa: F401


def oracle_rows(w, rows: torch.Tensor, nthreads: int = 0) -> np.ndarray:
    """The oracle's [n, k] result for the given rows of a workload."""
    win, L = gather_windows(w, rows)
    n, lmax = win.shape
    if w.row_to_batch is None:
        b = rows.cpu().numpy().astype(np.int32)
    else:
        b = w.row_to_batch[rows.to(w.row_to_batch.device)].cpu().numpy().astype(np.int32)
    table = w.page_table.reshape(-1).cpu().numpy()
    return topk_packed_reference(win.reshape(-1), lmax, L, np.zeros(n, np.int32), b, table,
                                 w.pt_stride, w.page_size, w.k, nthreads=nthreads)


def check_invariants_all_rows(w, out: torch.Tensor, chunk: int = 128) -> None:
    """Every row, on the device: count = min(k, L) in the prefix; outputs name
    pages of the row's own table row; window indices strictly ascending inside
    [0, L); every selected score >= every unselected one, ties to lower j."""
    dev = out.device
    k, P = w.k, w.page_size
    L = w.seq_lens.to(torch.int64).clamp_min(0)
    m = torch.minimum(L, torch.tensor(k, device=dev))
    slot = torch.arange(k, device=dev)
    taken = out >= 0
    assert torch.equal(taken, slot[None, :] < m[:, None]), "count / prefix of -1 padding"
    # inverse of the page transform (pages are distinct across the table)
    table = w.page_table.to(torch.int64)
    inv = torch.full((1 << 24,), -1, dtype=torch.int64, device=dev)
    cols = torch.arange(table.shape[1], device=dev)
    inv[table.reshape(-1)] = cols.repeat(table.shape[0])
    owner = torch.full((1 << 24,), -1, dtype=torch.int64, device=dev)
    owner[table.reshape(-1)] = torch.arange(table.shape[0], device=dev).repeat_interleave(table.shape[1])
    trow = w.table_rows().to(torch.int64)
    if w.row_to_batch is None and w.pt_stride == 0:
        trow = torch.zeros_like(trow)
    flat = w.scores.reshape(-1)
    for a in range(0, w.num_rows, chunk):
        o = out[a:a + chunk].to(torch.int64)
        t = taken[a:a + chunk]
        page = torch.where(t, o // P, torch.zeros_like(o))
        pidx = inv[page]
        assert bool(((pidx >= 0) | ~t).all()), "output names a page outside the table"
        assert bool(((owner[page] == trow[a:a + chunk, None]) | ~t).all()), "page of another table row"
        j = pidx * P + o % P
        Lc = L[a:a + chunk]
        assert bool((((j >= 0) & (j < Lc[:, None])) | ~t).all()), "index outside the window"
        asc = (j[:, 1:] > j[:, :-1]) | ~t[:, 1:]
        assert bool(asc.all()), "window indices not strictly ascending"
        # threshold property on rows with L > k
        big = Lc > k
        if not bool(big.any()):
            continue
        rows = torch.nonzero(big).flatten() + a
        lmax = int(L[rows].max().item())
        ar = torch.arange(lmax, device=dev)
        for b in range(0, rows.numel(), 16):
            rr = rows[b:b + 16]
            base = rr * w.row_stride + w.row_starts[rr].to(torch.int64)
            valid = ar[None, :] < L[rr][:, None]
            idx = torch.where(valid, base[:, None] + ar[None, :], torch.zeros_like(base[:, None]))
            vals = torch.where(valid, flat[idx], torch.full((1,), float("-inf"), device=dev))
            jj = j[rr - a]  # all k taken
            sel_vals = torch.gather(vals, 1, jj)
            lo = sel_vals.min(dim=1).values
            mask = torch.zeros_like(valid)
            mask.scatter_(1, jj, True)
            unsel = torch.where(mask | ~valid, torch.full((1,), float("-inf"), device=dev), vals)
            hi = unsel.max(dim=1).values
            assert bool((lo >= hi).all()), "a selected score is below an unselected one"
            tie = lo == hi
            if bool(tie.any()):
                big_idx = torch.full_like(vals, -1, dtype=torch.int64)
                arb = ar[None, :].expand_as(vals)
                sel_tied = torch.where(mask & (vals == lo[:, None]), arb, big_idx).max(dim=1).values
                uns_tied = torch.where(~mask & valid & (vals == lo[:, None]), arb,
                                       torch.full_like(big_idx, 1 << 40)).min(dim=1).values
                assert bool(((sel_tied < uns_tied) | ~tie).all()), "a tie went to a higher index"
