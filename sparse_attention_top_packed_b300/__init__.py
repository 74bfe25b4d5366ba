"""Packed-layout top-k + page transform for DSA sparse-attention prefill, on B300.

The operation (page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66% 끌어올린 Top-K
커널 최적화 분석", sglang PR #37889, Intro and sections 1-2): for each query row
i, take the score window scores[i, row_starts[i] : row_starts[i] + seq_lens[i]]
of a shared float32 buffer, select the k largest scores (a tie goes to the lower
window index), list the chosen window indices in ascending order, map each
through the row's page-table row, and pad with -1 when the window is shorter
than k.

The work is done by hand-written sm_103a CUDA behind a C ABI
(``include/topk_packed.h``, ``libtopk_packed.so``); :mod:`.binding` marshals
arguments to it.  There is no CPU path.
"""
from .binding import (  # noqa: F401
    TopkError,
    available,
    library_path,
    topk_packed,
    topk_packed_ex,
    topk_status_string,
)
