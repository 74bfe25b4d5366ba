"""Splitting one batch of rows over several GPUs (one process per GPU).

Rows are independent, so a batch shards by contiguous row ranges with no
exchange step: rank r runs ``topk_packed`` on rows ``[start, stop)`` by
passing pointer-offset slices of the per-row arrays, the score buffer and
the output (see :func:`row_range` and :func:`slice_args`).  Gathering the
outputs is left to the caller (one all-gather of ``[rows_r, k]`` int32 if
it wants them on one rank).
"""
from __future__ import annotations


def row_range(num_rows: int, rank: int, world: int) -> tuple[int, int]:
    """Rows ``[start, stop)`` of ``rank`` out of ``world``: contiguous, sizes
    differ by at most one, earlier ranks take the extra rows."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    if num_rows < 0:
        raise ValueError("num_rows must be >= 0")
    base, extra = divmod(num_rows, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def slice_args(scores, row_stride: int, seq_lens, row_starts, row_to_batch, out, start: int, stop: int):
    """The per-rank arguments for rows ``[start, stop)`` of a batch whose
    buffer has one score row per query row (the packed layout): tensors are
    sliced on their first dimension, so their data pointers move by whole
    rows.  ``row_to_batch`` may be None (identity): the identity map of the
    whole batch is then not the identity of the slice, so it is returned as
    an explicit range the caller must materialise."""
    sl = slice(start, stop)
    rtb = row_to_batch[sl] if row_to_batch is not None else None
    identity_offset = start if row_to_batch is None else None
    return scores[sl], seq_lens[sl], row_starts[sl], rtb, out[sl], identity_offset
