"""Seeded synthetic inputs for the packed top-k + page transform.

This module only draws inputs: score buffers, window lengths and offsets,
row -> table-row maps and page tables.  It holds none of the operation's
arithmetic, and both the library's tests/benchmark and the CPU oracle's tests
use it.

Layout of every problem (the packed DSA layout of the page "[sglang] [AMD
ROCm] GLM-5.x Prefill 성능을 66% 끌어올린 Top-K 커널 최적화 분석", Intro and
section 1): a float32 buffer of `rows x row_stride`; row i's window is
`scores[i*row_stride + row_starts[i] : ... + seq_lens[i]]`; row i uses page-table
row `row_to_batch[i]` (or i when the map is absent).

Named workloads (sizes of the sparse-attention prefill shapes this operator
serves):

  tiny         8 rows, buffer [8, 1024] N(0,1); seq_lens U{1..300}; row_starts
               U{0..700}; row_to_batch = i % 2; page table [2, 32]; page 64; k 32
  decode       64 rows, [64, 8192] N(0,1); seq_len 8192; row_starts 0; identity
               map (None); page table [64, 128]; page 64; k 2048
  prefill      two requests of 70000 KV tokens side by side (row_stride 140000);
               the last 2048 query tokens of each: row 2048*r + q has
               seq_len 67953 + q and row_start 70000*r, table row r; page table
               [2, 1094]; page 64; k 2048
  long         one request of 327680 KV tokens, its last 2048 query tokens:
               [2048, 327680], seq_len 325633 + q, row_start 0, every row on table
               row 0 (row_to_batch zeros); page table [1, 5120]; page 64; k 2048
  mixed        16 requests, KV lengths U{1024..65536} (seed 0), side by side;
               8192 query rows shared in proportion to length; the rows of a
               request sit at evenly spaced causal positions, so windows run
               from a few dozen tokens to the whole request (some shorter than
               k); scores N(0,1) rounded to bf16 and stored as float32 (ties);
               page table [16, 1024]; page 64; k 2048

Page tables hold distinct page numbers drawn without replacement from
[0, 2^24), so that page*64 + 63 < 2^31 and every output names its page.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import math

import numpy as np
import torch

PAGE_POOL = 1 << 24


@dataclass
class Workload:
    name: str
    scores: torch.Tensor          # [buffer_rows, row_stride] float32
    row_stride: int
    seq_lens: torch.Tensor        # [num_rows] int32
    row_starts: torch.Tensor      # [num_rows] int32
    row_to_batch: Optional[torch.Tensor]  # [num_rows] int32 or None (identity)
    page_table: torch.Tensor      # [table_rows, pt_stride] int32
    pt_stride: int
    page_size: int
    k: int
    num_rows: int

    @property
    def dtype(self) -> str:
        """Element type of the score buffer: "f32", "bf16" or "f16"."""
        return {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[self.scores.dtype]

    @property
    def elem_bytes(self) -> int:
        return self.scores.element_size()

    def window_bytes(self) -> int:
        """Bytes of the windows that must be read: rows with seq_len <= k need no scores."""
        L = self.seq_lens.to(torch.int64).clamp_min(0)
        return int((L * (L > self.k)).sum().item()) * self.elem_bytes

    def window_bytes_all(self) -> int:
        return int(self.seq_lens.to(torch.int64).clamp_min(0).sum().item()) * self.elem_bytes

    def output_bytes(self) -> int:
        return self.num_rows * self.k * 4

    def algorithmic_bytes(self) -> int:
        return self.window_bytes() + self.output_bytes()

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return Workload(self.name, mv(self.scores), self.row_stride, mv(self.seq_lens),
                        mv(self.row_starts), mv(self.row_to_batch), mv(self.page_table),
                        self.pt_stride, self.page_size, self.k, self.num_rows)

    def head(self, n: int) -> "Workload":
        """The first n query rows, with a copy of only the buffer rows they read
        (so the full buffer can be freed)."""
        n = min(int(n), self.num_rows)
        cut = lambda t: None if t is None else t[:n].clone()
        return Workload(self.name, self.scores[:n].clone(), self.row_stride, cut(self.seq_lens),
                        cut(self.row_starts), cut(self.row_to_batch), self.page_table,
                        self.pt_stride, self.page_size, self.k, n)

    def table_rows(self) -> torch.Tensor:
        """Table row of each query row (materialises the identity map)."""
        if self.row_to_batch is None:
            return torch.arange(self.num_rows, dtype=torch.int32, device=self.seq_lens.device)
        return self.row_to_batch


def with_dtype(w: Workload, dtype: str) -> Workload:
    """The same problem with the score buffer held as `dtype` ("f32", "bf16",
    "f16"): each value rounded to the nearest of the type (ties to even), by
    torch's conversion.  The layout, lengths, offsets and tables are shared."""
    t = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    return Workload(w.name, w.scores.to(t), w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch,
                    w.page_table, w.pt_stride, w.page_size, w.k, w.num_rows)


def distinct_pages(rows: int, cols: int, seed: int) -> torch.Tensor:
    """[rows, cols] int32 page numbers, all distinct, drawn from [0, 2^24)."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(PAGE_POOL, generator=g, dtype=torch.int64)[: rows * cols]
    return perm.to(torch.int32).reshape(rows, cols)


def _normal(shape, seed: int, device, bf16: bool = False) -> torch.Tensor:
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if bf16:
        x = x.to(torch.bfloat16).to(torch.float32)
    return x


def tiny(device="cpu", seed: int = 0) -> Workload:
    g = torch.Generator().manual_seed(seed)
    rows, stride = 8, 1024
    seq_lens = torch.randint(1, 301, (rows,), generator=g, dtype=torch.int64).to(torch.int32)
    row_starts = torch.randint(0, 701, (rows,), generator=g, dtype=torch.int64).to(torch.int32)
    rtb = (torch.arange(rows) % 2).to(torch.int32)
    pt = distinct_pages(2, 32, seed + 1)
    scores = _normal((rows, stride), seed, device)
    return Workload("tiny", scores, stride, seq_lens.to(device), row_starts.to(device),
                    rtb.to(device), pt.to(device), 32, 64, 32, rows)


def decode(device="cpu", seed: int = 0) -> Workload:
    rows, stride = 64, 8192
    scores = _normal((rows, stride), seed, device)
    seq_lens = torch.full((rows,), 8192, dtype=torch.int32)
    row_starts = torch.zeros(rows, dtype=torch.int32)
    pt = distinct_pages(64, 128, seed + 1)
    return Workload("decode", scores, stride, seq_lens.to(device), row_starts.to(device),
                    None, pt.to(device), 128, 64, 2048, rows)


def prefill(device="cpu", seed: int = 0, kv_len: int = 70000, q_per_req: int = 2048,
            requests: int = 2, k: int = 2048, page_size: int = 64) -> Workload:
    stride = kv_len * requests
    rows = q_per_req * requests
    q = torch.arange(q_per_req, dtype=torch.int64)
    seq_lens = torch.cat([kv_len - q_per_req + q + 1 for _ in range(requests)]).to(torch.int32)
    row_starts = torch.cat([torch.full((q_per_req,), kv_len * r, dtype=torch.int64)
                            for r in range(requests)]).to(torch.int32)
    rtb = torch.cat([torch.full((q_per_req,), r, dtype=torch.int64)
                     for r in range(requests)]).to(torch.int32)
    pages = -(-kv_len // page_size)
    pt = distinct_pages(requests, pages, seed + 1)
    scores = _normal((rows, stride), seed, device)
    return Workload("prefill", scores, stride, seq_lens.to(device), row_starts.to(device),
                    rtb.to(device), pt.to(device), pages, page_size, k, rows)


def long_context(device="cpu", seed: int = 0, kv_len: int = 327680, q_rows: int = 2048,
                 k: int = 2048, page_size: int = 64, identity_map: bool = False) -> Workload:
    """With identity_map=True the map is None and pt_stride is 0, so every row
    still reads table row 0 (the same result as the all-zero map)."""
    q = torch.arange(q_rows, dtype=torch.int64)
    seq_lens = (kv_len - q_rows + q + 1).to(torch.int32)
    row_starts = torch.zeros(q_rows, dtype=torch.int32)
    pages = -(-kv_len // page_size)
    pt = distinct_pages(1, pages, seed + 1)
    scores = _normal((q_rows, kv_len), seed, device)
    rtb = None if identity_map else torch.zeros(q_rows, dtype=torch.int32).to(device)
    return Workload("long", scores, kv_len, seq_lens.to(device), row_starts.to(device),
                    rtb, pt.to(device), 0 if identity_map else pages, page_size, k, q_rows)


def few_long(device="cpu", seed: int = 0, rows: int = 64, kv_len: int = 327680, k: int = 2048,
             page_size: int = 64) -> Workload:
    """Fewer rows than SMs with long windows (the case that splits a row over
    a cluster of CTAs): `rows` decode-like queries of one request of kv_len
    keys each, seeing the whole context, [rows, kv_len] N(0,1), one table row."""
    seq_lens = torch.full((rows,), kv_len, dtype=torch.int32)
    row_starts = torch.zeros(rows, dtype=torch.int32)
    pages = -(-kv_len // page_size)
    pt = distinct_pages(1, pages, seed + 1)
    scores = _normal((rows, kv_len), seed, device)
    return Workload("fewlong", scores, kv_len, seq_lens.to(device), row_starts.to(device),
                    torch.zeros(rows, dtype=torch.int32).to(device), pt.to(device), pages, page_size, k, rows)


def mixed_lengths(seed: int = 0, requests: int = 16, lo: int = 1024, hi: int = 65536):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (requests,), generator=g, dtype=torch.int64)


def mixed_rows(kv_lens: torch.Tensor, total_rows: int = 8192):
    """Rows per request in proportion to its length (floor, then one extra row
    per request in index order until the total is reached), at most the
    request's length."""
    L = kv_lens.to(torch.int64)
    total = int(L.sum())
    n = (total_rows * L) // total
    left = total_rows - int(n.sum())
    r = 0
    while left > 0:
        if n[r] < L[r]:
            n[r] += 1
            left -= 1
        r = (r + 1) % L.shape[0]
    return torch.minimum(n, L)


def mixed(device="cpu", seed_lengths: int = 0, seed_scores: int = 1, total_rows: int = 8192,
          requests: int = 16, lo: int = 1024, hi: int = 65536, k: int = 2048,
          page_size: int = 64, table_pages: int = 1024) -> Workload:
    L = mixed_lengths(seed_lengths, requests, lo, hi)
    n = mixed_rows(L, total_rows)
    offsets = torch.cumsum(L, 0) - L
    stride = int(L.sum())
    seq, starts, rtb = [], [], []
    for r in range(requests):
        q = torch.arange(1, int(n[r]) + 1, dtype=torch.int64)
        # evenly spaced causal positions: the q-th of n rows sees floor(q*L/n) keys
        seq.append((q * L[r]) // n[r])
        starts.append(torch.full((int(n[r]),), int(offsets[r]), dtype=torch.int64))
        rtb.append(torch.full((int(n[r]),), r, dtype=torch.int64))
    seq_lens = torch.cat(seq).to(torch.int32)
    row_starts = torch.cat(starts).to(torch.int32)
    row_to_batch = torch.cat(rtb).to(torch.int32)
    rows = int(seq_lens.shape[0])
    pages_needed = -(-int(L.max()) // page_size)
    if pages_needed > table_pages:
        raise ValueError("page table too narrow for the longest request")
    pt = distinct_pages(requests, table_pages, seed_lengths + 2)
    scores = _normal((rows, stride), seed_scores, device, bf16=True)
    return Workload("mixed", scores, stride, seq_lens.to(device), row_starts.to(device),
                    row_to_batch.to(device), pt.to(device), table_pages, page_size, k, rows)


def prefill_drift(device="cpu", seed: int = 0, period_mean: float = 300.0, period_scale: float = 450.0,
                  jitter: float = 0.05) -> Workload:
    """The prefill shape with scores whose distribution moves from row to row,
    as an indexer's scores do along the queries of a request: row q of a
    request (its q-th causal query) holds N(0,1) * s_q + m_q with
      m_q = 0.5 sin(2 pi q / period_mean) + jitter * N(0,1)   (seeded),
      s_q = 1 + 0.25 sin(2 pi q / period_scale).
    Neighbouring rows differ by about 0.01 of a standard deviation in the mean
    plus the jitter, so a threshold carried from one row to the next is often
    too high or too low."""
    w = prefill(device=device, seed=seed)
    q_per_req = w.num_rows // 2
    q = torch.arange(w.num_rows, dtype=torch.float64) % q_per_req
    g = torch.Generator().manual_seed(seed + 7)
    m = 0.5 * torch.sin(2 * math.pi * q / period_mean) + jitter * torch.randn(w.num_rows, generator=g,
                                                                                dtype=torch.float64)
    sc = 1.0 + 0.25 * torch.sin(2 * math.pi * q / period_scale)
    w.scores.mul_(sc.to(torch.float32).to(w.scores.device)[:, None]).add_(m.to(torch.float32).to(w.scores.device)[:, None])
    w.name = "drift"
    return w


NAMED = {"tiny": tiny, "decode": decode, "prefill": prefill, "long": long_context, "mixed": mixed,
         "fewlong": few_long, "drift": prefill_drift}


def named(name: str, device="cpu", **kw) -> Workload:
    return NAMED[name](device=device, **kw)


# ---------------------------------------------------------------------------
# Host copies of windows (for the CPU oracle in tests and the benchmark's
# CPU-baseline leg).
# ---------------------------------------------------------------------------

def gather_windows(w: Workload, rows: torch.Tensor, chunk: int = 256):
    """Host float32 [n, Lmax] windows of `rows` (padded with +inf) and their lengths."""
    rows = rows.to(torch.int64).to(w.seq_lens.device)
    L = w.seq_lens[rows].to(torch.int64).clamp_min(0)
    starts = w.row_starts[rows].to(torch.int64)
    lmax = max(int(L.max().item()) if rows.numel() else 0, 1)
    flat = w.scores.reshape(-1)
    out = np.empty((rows.numel(), lmax), dtype=np.float32)
    ar = torch.arange(lmax, device=flat.device, dtype=torch.int64)
    for a in range(0, rows.numel(), chunk):
        r = rows[a:a + chunk]
        base = r * w.row_stride + starts[a:a + chunk]
        valid = ar[None, :] < L[a:a + chunk, None]
        idx = torch.where(valid, base[:, None] + ar[None, :], torch.zeros_like(base[:, None]))
        vals = flat[idx].float()
        vals = torch.where(valid, vals, torch.full_like(vals, float("inf")))
        out[a:a + r.numel()] = vals.cpu().numpy()
    return out, L.cpu().numpy().astype(np.int32)


def sample_rows(num_rows: int, n: int, seed: int = 0) -> torch.Tensor:
    """Deterministic sample: the first and last rows plus evenly spread random ones."""
    if num_rows <= n:
        return torch.arange(num_rows)
    g = torch.Generator().manual_seed(seed)
    edge = min(32, n // 4)
    mid = torch.randperm(num_rows - 2 * edge, generator=g)[: n - 2 * edge] + edge
    return torch.cat([torch.arange(edge), torch.sort(mid).values,
                      torch.arange(num_rows - edge, num_rows)])


# ---------------------------------------------------------------------------
# Small random problems for parity sweeps and oracle pins (host numpy arrays).
# ---------------------------------------------------------------------------

TIE_VALUES = np.array([-2.0, -1.0, -0.0, 0.0, 1.0, 2.0, np.inf, -np.inf], dtype=np.float32)


@dataclass
class HostProblem:
    scores: np.ndarray        # float32 [rows * row_stride]
    row_stride: int
    seq_lens: np.ndarray      # int32 [rows]
    row_starts: np.ndarray    # int32 [rows]
    row_to_batch: Optional[np.ndarray]
    page_table: np.ndarray    # int32 [table_rows * pt_stride]
    pt_stride: int
    page_size: int
    k: int

    @property
    def num_rows(self) -> int:
        return int(self.seq_lens.shape[0])


def random_problem(rng: np.random.Generator, rows: int, max_len: int, k: int, page_size: int,
                   values: str = "normal", slack: int = 16, identity: bool = False,
                   table_rows: Optional[int] = None, forced_lens=None) -> HostProblem:
    """A packed problem with ragged, unaligned windows.

    values: "normal" (N(0,1)), "ties" (drawn from TIE_VALUES, incl. +-0, +-inf),
    "bf16" (N(0,1) rounded to bf16), "equal" (one constant), "int" (small
    integers: heavy ties), "ascending"/"descending" (sorted windows).
    Cells outside the windows hold +inf so that a read outside a window shows.
    """
    row_stride = max_len + slack
    if forced_lens is not None:
        seq_lens = np.asarray(forced_lens, dtype=np.int64)[:rows]
    else:
        seq_lens = rng.integers(0, max_len + 1, size=rows)
    row_starts = np.array([rng.integers(0, row_stride - max(L, 0) + 1) for L in seq_lens])
    scores = np.full(rows * row_stride, np.inf, dtype=np.float32)
    for i in range(rows):
        L = int(max(seq_lens[i], 0))
        if values == "normal":
            w = rng.standard_normal(L).astype(np.float32)
        elif values == "ties":
            w = TIE_VALUES[rng.integers(0, TIE_VALUES.shape[0], size=L)]
        elif values == "bf16":
            w = _round_bf16(rng.standard_normal(L).astype(np.float32))
        elif values == "equal":
            w = np.full(L, 0.25, dtype=np.float32)
        elif values == "int":
            w = rng.integers(-3, 4, size=L).astype(np.float32)
        elif values == "ascending":
            w = np.sort(rng.standard_normal(L).astype(np.float32))
        elif values == "descending":
            w = np.sort(rng.standard_normal(L).astype(np.float32))[::-1].copy()
        else:
            raise ValueError(values)
        base = i * row_stride + int(row_starts[i])
        scores[base: base + L] = w
    pages_per_row = max(1, -(-max_len // page_size))
    if identity:
        n_table = rows
        rtb = None
    else:
        n_table = table_rows if table_rows is not None else max(1, rows // 3)
        rtb = rng.integers(0, n_table, size=rows).astype(np.int32)
    pool = rng.choice(PAGE_POOL, size=n_table * pages_per_row, replace=False).astype(np.int32)
    return HostProblem(scores, row_stride, seq_lens.astype(np.int32), row_starts.astype(np.int32),
                       rtb, pool, pages_per_row, page_size, k)


def _round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bf16 (ties to even) -> float32, on the bit pattern."""
    u = x.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    u = ((u + rounding) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)
