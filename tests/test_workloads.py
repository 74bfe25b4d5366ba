"""The synthetic configurations' shapes and the benchmark's byte accounting
(no GPU; the score buffers are replaced by a stub, only the row layout and the
page tables are built).

The expected byte counts follow from the configurations' definitions by hand:
prefill, rows 2048 r + q with L = 67953 + q (q < 2048) in each of 2 requests,
reads sum(L) * 4 = 2 * 4 * (2048 * 67953 + 2047 * 2048 / 2) = 1,130,110,976 bytes
and writes 4096 * 2048 * 4 = 33,554,432; long, L = 325633 + q over 2048 rows,
reads 4 * (2048 * 325633 + 2047 * 2048 / 2) = 2,675,970,048 and writes
2048 * 2048 * 4 = 16,777,216; decode reads 64 * 8192 * 4 and writes 64 * 2048 * 4.
"""
import pytest
import torch

from sparse_attention_top_packed_b300 import workloads as wl


@pytest.fixture
def no_scores(monkeypatch):
    monkeypatch.setattr(wl, "_normal", lambda shape, seed, device, bf16=False: torch.zeros((1, 1)))


def test_prefill_layout_and_bytes(no_scores):
    w = wl.prefill(device="cpu")
    assert w.num_rows == 4096 and w.row_stride == 140000 and w.k == 2048 and w.page_size == 64
    L = w.seq_lens.to(torch.int64)
    assert int(L.min()) == 67953 and int(L.max()) == 70000
    assert torch.equal(w.seq_lens[:2048], w.seq_lens[2048:])
    assert set(w.row_starts.tolist()) == {0, 70000}
    assert (w.row_starts.to(torch.int64) + L <= w.row_stride).all()
    assert w.page_table.shape == (2, 1094)
    assert w.window_bytes() == 1_130_110_976
    assert w.output_bytes() == 33_554_432
    assert w.algorithmic_bytes() == 1_163_665_408


def test_long_context_layout_and_bytes(no_scores):
    w = wl.long_context(device="cpu")
    assert w.num_rows == 2048 and w.row_stride == 327680
    L = w.seq_lens.to(torch.int64)
    assert int(L.min()) == 325633 and int(L.max()) == 327680
    assert w.page_table.shape == (1, 5120)
    assert int(w.row_to_batch.abs().sum()) == 0  # one request: every row uses table row 0
    assert w.window_bytes() == 2_675_970_048 and w.output_bytes() == 16_777_216


def test_decode_bytes(no_scores):
    w = wl.decode(device="cpu")
    assert w.algorithmic_bytes() == 64 * 8192 * 4 + 64 * 2048 * 4


def test_rows_no_longer_than_k_read_nothing(no_scores):
    w = wl.tiny(device="cpu")
    L = w.seq_lens.to(torch.int64).clamp_min(0)
    assert w.window_bytes() == int((L * (L > w.k)).sum()) * 4
    assert w.window_bytes_all() == int(L.sum()) * 4


def test_pages_are_distinct_and_fit_31_bits():
    t = wl.distinct_pages(16, 1024, 3)
    flat = t.reshape(-1)
    assert flat.unique().numel() == flat.numel()
    assert int(flat.max()) * 64 + 63 < 2 ** 31


def test_drift_recipe(monkeypatch):
    """Each row is N(0,1) * s_q + m_q; with the normal draw stubbed to ones a
    row holds s_q + m_q, whose smooth part follows the stated sines and whose
    rest is the 0.05-sigma jitter."""
    import math

    monkeypatch.setattr(wl, "_normal", lambda shape, seed, device, bf16=False: torch.ones((shape[0], 1)))
    w = wl.prefill_drift(device="cpu")
    q = torch.arange(w.num_rows, dtype=torch.float64) % 2048
    smooth = 1.0 + 0.25 * torch.sin(2 * math.pi * q / 450) + 0.5 * torch.sin(2 * math.pi * q / 300)
    rest = w.scores[:, 0].to(torch.float64) - smooth
    assert abs(float(rest.mean())) < 0.005 and 0.045 < float(rest.std()) < 0.055
    assert w.name == "drift" and w.num_rows == 4096 and w.row_stride == 140000
