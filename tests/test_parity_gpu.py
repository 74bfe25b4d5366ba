"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bit-exact int32 equality everywhere (the result is unique).  Small problems are
compared element by element for every kernel path; the full-size workloads, in
the launch the benchmark times, are compared row by row on a sample of rows
and checked on every row for the invariants of the result."""
import zlib

import numpy as np
import pytest
import torch

from oracle import topk_packed_reference
from sparse_attention_top_packed_b300 import binding
from sparse_attention_top_packed_b300 import workloads as wl
from tests.gpu_helpers import check_invariants_all_rows, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

PATHS = [dict(path="pipe"), dict(path="split"), dict(path="multipass"), dict(path="stream", cluster_size=1),
         dict(path="stream", cluster_size=2), dict(path="stream", cluster_size=4),
         dict(path="stream", cluster_size=8)]
PATH_IDS = ["pipe", "split", "multipass", "stream1", "stream2", "stream4", "stream8"]


def run(w, **launch):
    out = torch.full((w.num_rows, w.k), -7, dtype=torch.int32, device=w.scores.device)
    binding.run_workload(w, out=out, **launch)
    torch.cuda.synchronize()
    return out


def host_problem_to_device(p, dev):
    rows = p.num_rows
    return wl.Workload("random", torch.from_numpy(p.scores).to(dev).reshape(rows, p.row_stride),
                       p.row_stride, torch.from_numpy(p.seq_lens).to(dev),
                       torch.from_numpy(p.row_starts).to(dev),
                       None if p.row_to_batch is None else torch.from_numpy(p.row_to_batch).to(dev),
                       torch.from_numpy(p.page_table).to(dev), p.pt_stride, p.page_size, p.k, rows)


def oracle_host(p):
    return topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch,
                                 p.page_table, p.pt_stride, p.page_size, p.k)


@pytest.fixture(autouse=True)
def _flags_stay_clear(cuda_device):
    binding.topk_packed_device_flags(reset=True)
    yield
    assert binding.topk_packed_device_flags() == 0, "a bounded device wait gave up"


@pytest.mark.parametrize("launch", PATHS, ids=PATH_IDS)
def test_tiny(cuda_device, launch):
    w = wl.tiny(device=cuda_device)
    out = run(w, **launch)
    want = oracle_rows(w, torch.arange(w.num_rows))
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("launch", PATHS, ids=PATH_IDS)
def test_decode(cuda_device, launch):
    w = wl.decode(device=cuda_device)
    out = run(w, **launch)
    want = oracle_rows(w, torch.arange(w.num_rows))
    assert np.array_equal(out.cpu().numpy(), want)
    check_invariants_all_rows(w, out)


CASES = [
    # values, rows, max_len, k, page_size
    ("normal", 24, 20000, 2048, 64),
    ("normal", 40, 9000, 300, 16),
    ("bf16", 24, 30000, 2048, 64),
    ("ties", 30, 12000, 777, 1),
    ("int", 16, 20000, 2048, 64),
    ("equal", 8, 10000, 2048, 64),
    ("ascending", 10, 25000, 2048, 64),
    ("descending", 10, 25000, 2048, 64),
    ("normal", 20, 5000, 1, 4),
    ("normal", 12, 70000, 2048, 64),
    ("bf16", 50, 3000, 32, 64),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-L{c[2]}-k{c[3]}" for c in CASES])
@pytest.mark.parametrize("launch", PATHS, ids=PATH_IDS)
def test_random_problems(cuda_device, case, launch):
    values, rows, max_len, k, page_size = case
    rng = np.random.default_rng(zlib.crc32(f"{values}-{max_len}-{k}".encode()))
    p = wl.random_problem(rng, rows=rows, max_len=max_len, k=k, page_size=page_size, values=values,
                          slack=13)
    w = host_problem_to_device(p, cuda_device)
    before = w.scores.clone()
    out = run(w, **launch)
    assert torch.equal(before, w.scores), "the score buffer was written"
    assert np.array_equal(out.cpu().numpy(), oracle_host(p))


@pytest.mark.parametrize("launch", PATHS, ids=PATH_IDS)
def test_edge_lengths_and_offsets(cuda_device, launch):
    """seq_len in {0, 1, k-1, k, k+1, a tile boundary +-1}, every start offset
    mod 4, an odd row stride (so absolute alignment differs from row_start % 4),
    identity map, signed zeros and infinities in the windows."""
    k = 64
    lens = [0, 1, k - 1, k, k + 1, 4095, 4096, 4097, 8191, 8193, 2 * 4096 * 8 + 3, -5]
    rng = np.random.default_rng(3)
    rows = []
    for L in lens:
        for off in range(4):
            rows.append((L, off))
    n = len(rows)
    stride = max(L for L, _ in rows) + 7
    stride += 1 - stride % 2  # odd: absolute alignment differs from row_start % 4
    scores = np.full(n * stride, np.inf, dtype=np.float32)
    seq = np.zeros(n, np.int32)
    st = np.zeros(n, np.int32)
    for i, (L, off) in enumerate(rows):
        Lp = max(L, 0)
        v = rng.standard_normal(Lp).astype(np.float32)
        if Lp > 10:
            v[rng.integers(0, Lp, size=Lp // 10)] = -0.0
            v[rng.integers(0, Lp, size=Lp // 10)] = 0.0
            v[rng.integers(0, Lp, size=3)] = np.inf
            v[rng.integers(0, Lp, size=3)] = -np.inf
        seq[i] = L
        st[i] = off + (i % 3)
        scores[i * stride + st[i]: i * stride + st[i] + Lp] = v
    pages = -(-stride // 16)
    table = rng.choice(1 << 24, size=n * pages, replace=False).astype(np.int32)
    p = wl.HostProblem(scores, stride, seq, st, None, table, pages, 16, k)
    w = host_problem_to_device(p, cuda_device)
    out = run(w, **launch)
    assert np.array_equal(out.cpu().numpy(), oracle_host(p))


@pytest.mark.parametrize("k", [1, 2, 31, 512, 2048])
def test_k_values_against_each_other_and_oracle(cuda_device, k):
    rng = np.random.default_rng(k)
    p = wl.random_problem(rng, rows=16, max_len=12000, k=k, page_size=64, values="bf16")
    w = host_problem_to_device(p, cuda_device)
    want = oracle_host(p)
    for launch in PATHS:
        assert np.array_equal(run(w, **launch).cpu().numpy(), want), launch


def test_non_default_stream(cuda_device):
    w = wl.tiny(device=cuda_device)
    s = torch.cuda.Stream()
    out = torch.empty((w.num_rows, w.k), dtype=torch.int32, device=cuda_device)
    with torch.cuda.stream(s):
        binding.run_workload(w, out=out, stream=s)
    s.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle_rows(w, torch.arange(w.num_rows)))


def test_zero_rows_launches_nothing(cuda_device):
    w = wl.tiny(device=cuda_device)
    out = torch.full((1,), 5, dtype=torch.int32, device=cuda_device)
    binding.topk_packed(w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch,
                        w.page_table, w.pt_stride, w.page_size, w.k, out, 0)
    torch.cuda.synchronize()
    assert out.item() == 5


def test_plan_reports_the_launch(cuda_device):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = binding.topk_packed_plan(140000, 2048, 4096)
    assert plan["path"] == binding.PATHS["split"]
    assert plan["threads_per_cta"] == 512, "8 streaming and 8 finishing warps"
    assert plan["grid_ctas"] == sms, "one CTA per SM"
    small = binding.topk_packed_plan(140000, 2048, sms // 2 + 7)
    assert small["grid_ctas"] == sms // 2 + 7 and small["path"] == binding.PATHS["split"]
    dec = binding.topk_packed_plan(8192, 2048, 64)
    assert dec["path"] == binding.PATHS["decode"] and dec["grid_ctas"] == 64 and dec["threads_per_cta"] == 1024
    assert binding.topk_packed_plan(binding.DECODE_MAX_STRIDE, 2048, 64)["path"] == binding.PATHS["decode"]
    assert binding.topk_packed_plan(binding.DECODE_MAX_STRIDE + 1, 2048, 64)["path"] == binding.PATHS["split"]
    few = binding.topk_packed_plan(327680, 2048, sms // 2)
    assert few["path"] == binding.PATHS["stream"] and few["cluster_size"] == 2, "few long rows: 2-CTA clusters"
    fewer = binding.topk_packed_plan(327680, 2048, sms // 4)
    assert fewer["path"] == binding.PATHS["stream"] and fewer["cluster_size"] == 4
    assert binding.topk_packed_plan(327680, 2048, sms // 2 + 1)["path"] == binding.PATHS["split"]
    assert binding.topk_packed_plan(65535, 2048, 8)["path"] == binding.PATHS["split"]
    pipe = binding.topk_packed_plan(140000, 2048, 4096, path="pipe")
    assert pipe["threads_per_cta"] == 256, "8 warps, each streaming its own block"
    assert pipe["grid_ctas"] == 2 * sms, "two pipelined CTAs per SM"
    st = binding.topk_packed_plan(140000, 2048, 4096, path="stream")
    assert st["threads_per_cta"] == 1024
    assert st["grid_ctas"] % st["cluster_size"] == 0
    mp = binding.topk_packed_plan(140000, 2048, 4096, path="multipass")
    assert mp["path"] == binding.PATHS["multipass"]


# ---------------------------------------------------------------------------
# Full-size workloads, in the launch the benchmark times (topk_packed, auto).
# ---------------------------------------------------------------------------
def _full_size(w, sample: int):
    out = torch.empty((w.num_rows, w.k), dtype=torch.int32, device=w.scores.device)
    checksum = w.scores.view(torch.int32).sum(dtype=torch.int64)
    binding.topk_packed(w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch,
                        w.page_table, w.pt_stride, w.page_size, w.k, out, w.num_rows)
    torch.cuda.synchronize()
    assert torch.equal(checksum, w.scores.view(torch.int32).sum(dtype=torch.int64))
    rows = sample_rows(w.num_rows, sample)
    want = oracle_rows(w, rows)
    got = out[rows.to(out.device)].cpu().numpy()
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, f"rows {rows[bad[:10]].tolist()} differ from the oracle"
    check_invariants_all_rows(w, out)
    return out


def test_prefill_full_size(cuda_device):
    w = wl.prefill(device=cuda_device)
    out = _full_size(w, sample=512)
    # the cluster path gives the same bits
    out2 = run(w, path="stream", cluster_size=2)
    assert torch.equal(out, out2)
    assert torch.equal(out, run(w, path="split"))


def test_prefill_with_drifting_scores_full_size(cuda_device):
    """Rows whose score distribution moves from row to row: carried thresholds
    miss in both directions, and the rows they miss are redone exactly."""
    w = wl.prefill_drift(device=cuda_device)
    out = _full_size(w, sample=384)
    assert torch.equal(out, run(w, path="pipe"))


def test_long_context_full_size(cuda_device):
    w = wl.long_context(device=cuda_device)
    out = _full_size(w, sample=160)
    wi = wl.long_context(device=cuda_device, identity_map=True)
    out_id = run(wi)
    assert torch.equal(out, out_id), "row_to_batch=NULL with pt_stride 0 must match the zero map"
    out4 = run(w, path="stream", cluster_size=4)
    assert torch.equal(out, out4)
    assert torch.equal(out, run(w, path="split"))


def test_mixed_full_size(cuda_device):
    w = wl.mixed(device=cuda_device)
    assert int((w.seq_lens < w.k).sum()) > 0, "the mixed batch must hold windows shorter than k"
    out = _full_size(w, sample=768)
    out2 = run(w, path="multipass")
    assert torch.equal(out, out2)
    assert torch.equal(out, run(w, path="split"))


# ---------------------------------------------------------------------------
# The pipelined kernel carries an admission threshold from one row of a CTA to
# the next.  With one or two CTAs every row follows another in the same CTA,
# so these sequences drive each branch: a hint above the next row's k-th key
# (the row is streamed again), a hint far below it (the candidate buffer is
# compacted), ties across the threshold (exact compaction on (key, index)),
# rows much shorter or longer than the previous one, and rows whose k-th
# largest score is -inf.
# ---------------------------------------------------------------------------
def _sequence_problem(rng, kind, rows=12, L=20000, k=2048, page_size=64):
    stride = L + 37
    scores = np.full(rows * stride, np.inf, dtype=np.float32)
    seq = np.zeros(rows, np.int32)
    st = np.zeros(rows, np.int32)
    for i in range(rows):
        n = L
        if kind == "lengths":
            n = [L, L // 6, L, 3000, L, 2100, L // 2, L][i % 8]
        base = rng.standard_normal(n).astype(np.float32)
        if kind == "falling":      # each row's scores sit below the previous row's
            v = base - 0.5 * i
        elif kind == "rising":     # each row's scores sit above the previous row's
            v = base + 0.75 * i
        elif kind == "ties":       # few distinct values: big tie groups at every threshold
            v = np.round(base * 2.0) / 2.0
        elif kind == "neg_inf":    # most of the window is -inf: the k-th largest is -inf
            v = base.copy()
            v[rng.random(n) < 0.97] = -np.inf
        elif kind == "ramp":       # ascending windows: every chunk beats everything before it
            v = np.sort(base)
        else:
            v = base
        seq[i] = n
        st[i] = int(rng.integers(0, stride - n + 1))
        scores[i * stride + st[i]: i * stride + st[i] + n] = v.astype(np.float32)
    pages = -(-stride // page_size)
    table = rng.choice(1 << 24, size=2 * pages, replace=False).astype(np.int32)
    rtb = (np.arange(rows) % 2).astype(np.int32)
    return wl.HostProblem(scores, stride, seq, st, rtb, table, pages, page_size, k)


@pytest.mark.parametrize("kind", ["falling", "rising", "ties", "neg_inf", "ramp", "lengths"])
@pytest.mark.parametrize("ctas", [1, 2])
@pytest.mark.parametrize("path", ["pipe", "split"])
def test_pipe_threshold_carried_between_rows(cuda_device, kind, ctas, path):
    rng = np.random.default_rng(zlib.crc32(kind.encode()))
    p = _sequence_problem(rng, kind)
    w = host_problem_to_device(p, cuda_device)
    want = oracle_host(p)
    got = run(w, path=path, max_ctas=ctas).cpu().numpy()
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, f"rows {bad.tolist()} differ"


@pytest.mark.parametrize("lo,hi", [(2300, 6000), (3900, 4400), (2100, 2600)])
@pytest.mark.parametrize("ctas", [1, 2])
@pytest.mark.parametrize("path", ["pipe", "split"])
def test_short_bf16_rows_in_sequence(cuda_device, lo, hi, ctas, path):
    """Rows a little longer than k with bf16-rounded scores, one after another
    on one or two CTAs (thresholds carried from row to row): the k-th largest
    sits where bins of keys hold many distinct values, so the selection's
    first fine level meets crowded bins of several keys and its second level
    (or the generic selection) settles them."""
    rng = np.random.default_rng(lo * 7 + hi)
    lens = rng.integers(lo, hi + 1, size=48)
    p = wl.random_problem(rng, rows=48, max_len=hi, k=2048, page_size=64, values="bf16", slack=5,
                          forced_lens=lens)
    w = host_problem_to_device(p, cuda_device)
    got = run(w, path=path, max_ctas=ctas).cpu().numpy()
    bad = np.nonzero((got != oracle_host(p)).any(axis=1))[0]
    assert bad.size == 0, f"rows {bad.tolist()} differ"


RAW_CASES = [
    # values, rows, max_len, k: several rows per CTA on one or two CTAs, windows
    # shorter than k among them, so the row-to-row paths run without a table
    ("normal", 12, 20000, 2048),
    ("bf16", 16, 9000, 512),
    ("ties", 10, 3000, 2048),
]


@pytest.mark.parametrize("case", RAW_CASES, ids=[f"{c[0]}-L{c[2]}-k{c[3]}" for c in RAW_CASES])
@pytest.mark.parametrize("launch", PATHS + [dict(path="pipe", max_ctas=2)], ids=PATH_IDS + ["pipe2"])
def test_raw_indices_without_page_table(cuda_device, case, launch):
    values, rows, max_len, k = case
    rng = np.random.default_rng(zlib.crc32(f"raw-{values}-{max_len}".encode()))
    p = wl.random_problem(rng, rows=rows, max_len=max_len, k=k, page_size=64, values=values, slack=9)
    w = host_problem_to_device(p, cuda_device)
    out = torch.full((w.num_rows, k), -7, dtype=torch.int32, device=cuda_device)
    binding.topk_packed_ex(w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch, None,
                           0, 0, k, out, w.num_rows, **launch)
    torch.cuda.synchronize()
    want = topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch,
                                 None, 0, 1, k)
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("launch", PATHS, ids=PATH_IDS)
def test_kth_largest_is_negative_infinity(cuda_device, launch):
    rng = np.random.default_rng(11)
    p = _sequence_problem(rng, "neg_inf", rows=6, L=9000, k=512)
    w = host_problem_to_device(p, cuda_device)
    assert np.array_equal(run(w, **launch).cpu().numpy(), oracle_host(p))


@pytest.mark.parametrize("name", ["long", "prefill"])
@pytest.mark.parametrize("path", ["auto", "split"])
def test_repeated_launches_are_identical(cuda_device, name, path):
    """The ring's stages are refilled by TMA while other warps may still be
    finishing a row: any ordering mistake between the consumers' reads and the
    next copy shows up as launch-to-launch differences."""
    w = wl.named(name, device=cuda_device)
    first = run(w, path=path)
    for _ in range(3):
        assert torch.equal(first, run(w, path=path)), "two launches on the same input disagree"


# ---------------------------------------------------------------------------
# The give-up path of a bounded wait, made to run on purpose: each streaming
# warp first waits on a barrier that nothing completes, with a 50 us bound.
# The wait runs out, bit 0 of the diagnostics word is raised, the warps stop
# taking chunks, the rows are finished exactly from global memory, and every
# copy already issued is waited for before the kernel exits.  Nothing faults:
# the result must still be the oracle's, and the next normal call too.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", ["pipe", "split"])
def test_stream_wait_give_up_is_recorded_and_the_result_stays_exact(cuda_device, path):
    rng = np.random.default_rng(77)
    p = wl.random_problem(rng, rows=24, max_len=20000, k=2048, page_size=64, values="normal", slack=13)
    w = host_problem_to_device(p, cuda_device)
    want = oracle_host(p)
    binding.topk_packed_device_flags(reset=True)
    out = torch.full((w.num_rows, w.k), -7, dtype=torch.int32, device=cuda_device)
    binding.topk_packed_ex(w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch, w.page_table,
                           w.pt_stride, w.page_size, w.k, out, w.num_rows, path=path, stream_wait_ns=50_000,
                           test_flags=binding.TEST_UNSATISFIED_WAIT)
    torch.cuda.synchronize()
    flags = binding.topk_packed_device_flags(reset=True)
    assert flags & 1, "the wait that nothing completes must be recorded as given up"
    assert np.array_equal(out.cpu().numpy(), want)
    assert np.array_equal(run(w, path=path).cpu().numpy(), want)


# ---------------------------------------------------------------------------
# Dependent launch (page section 2: the top-k kernel waits on the grid that
# produced its scores).  The producer lets its dependents start at once, waits
# 100 us, then writes the real scores over a buffer holding their negation.
# A top-k kernel that read a score before its wait returned would select from
# the negated values.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("launch", [dict(path="split"), dict(path="pipe"), dict(path="multipass"),
                                    dict(path="stream", cluster_size=2), dict(path="decode")],
                         ids=["split", "pipe", "multipass", "stream2", "decode"])
def test_dependent_launch_waits_for_the_producing_kernel(cuda_device, launch):
    from sparse_attention_top_packed_b300.producer import produce_scores

    rng = np.random.default_rng(5)
    p = wl.random_problem(rng, rows=24, max_len=16000, k=2048, page_size=64, values="normal", slack=13)
    w = host_problem_to_device(p, cuda_device)
    real = w.scores.clone()
    want = oracle_host(p)
    stream = torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(stream):
            w.scores.copy_(-real)
        out = torch.full((w.num_rows, w.k), -7, dtype=torch.int32, device=cuda_device)
        produce_scores(w.scores, real, delay_ns=100_000, stream=stream)
        binding.topk_packed_ex(w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch, w.page_table,
                               w.pt_stride, w.page_size, w.k, out, w.num_rows, dependent_launch=True,
                               stream=stream, **launch)
        stream.synchronize()
        assert np.array_equal(out.cpu().numpy(), want)


# ---------------------------------------------------------------------------
# k above the single-pass kernels' size (2048): the automatic choice is the
# multipass kernel; the stream kernel also serves it; pipe and split refuse.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("k", [2049, 4096, 10000])
def test_large_k(cuda_device, k):
    rng = np.random.default_rng(k + 17)
    p = wl.random_problem(rng, rows=12, max_len=30000, k=k, page_size=64, values="bf16", slack=11,
                          forced_lens=[30000, 20000, k + 1, k, k - 1, 0, 12345, 29999, min(4 * k, 30000), 1, 7777, 25000])
    w = host_problem_to_device(p, cuda_device)
    want = oracle_host(p)
    assert binding.topk_packed_plan(w.row_stride, k, w.num_rows)["path"] == binding.PATHS["multipass"]
    assert np.array_equal(run(w).cpu().numpy(), want)
    assert np.array_equal(run(w, path="stream", cluster_size=2).cpu().numpy(), want)
    for path in ("pipe", "split"):
        with pytest.raises(binding.TopkError):
            run(w, path=path)


# ---------------------------------------------------------------------------
# 16-bit score buffers (bfloat16, IEEE binary16).  The oracle reads the same
# bit patterns; ragged windows at every element offset (a 16-byte quad holds 8
# elements, so the head runs 0..7), odd strides, tie-heavy and special values.
# ---------------------------------------------------------------------------
def _half_host_problem(rng, dtype, rows, max_len, k, values):
    p = wl.random_problem(rng, rows=rows, max_len=max_len, k=k, page_size=64, values=values, slack=29)
    t = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    half = torch.from_numpy(p.scores).to(t)  # rounded to the type; +inf outside the windows stays +inf
    return p, half


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("values,rows,max_len,k", [("normal", 24, 20000, 2048), ("ties", 30, 9000, 300),
                                                   ("int", 16, 20000, 2048), ("normal", 40, 5000, 1),
                                                   ("bf16", 50, 3000, 32), ("equal", 8, 10000, 2048),
                                                   ("ascending", 10, 25000, 2048)])
def test_half_width_random_problems(cuda_device, dtype, values, rows, max_len, k):
    rng = np.random.default_rng(zlib.crc32(f"{dtype}-{values}-{max_len}-{k}".encode()))
    p, half = _half_host_problem(rng, dtype, rows, max_len, k, values)
    w = wl.Workload("random", half.to(cuda_device).reshape(rows, p.row_stride), p.row_stride,
                    torch.from_numpy(p.seq_lens).to(cuda_device), torch.from_numpy(p.row_starts).to(cuda_device),
                    torch.from_numpy(p.row_to_batch).to(cuda_device), torch.from_numpy(p.page_table).to(cuda_device),
                    p.pt_stride, p.page_size, p.k, rows)
    before = w.scores.clone()
    out = run(w)
    assert torch.equal(before, w.scores), "the score buffer was written"
    bits = half.view(torch.int16).numpy().view(np.uint16)
    want = topk_packed_reference(bits, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch, p.page_table,
                                 p.pt_stride, p.page_size, p.k, dtype=dtype)
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_half_width_edge_lengths_offsets_and_specials(cuda_device, dtype):
    """Every element offset mod 8, an odd stride, lengths around k and around
    the chunk sizes, signed zeros, infinities and (binary16) subnormals."""
    k = 64
    lens = [0, 1, k - 1, k, k + 1, 2047, 2048, 2049, 8191, 8193, 3 * 2048 * 8 + 5, -3]
    rng = np.random.default_rng(31)
    rows = [(L, off) for L in lens for off in range(8)]
    n = len(rows)
    stride = max(L for L, _ in rows) + 11
    stride += 1 - stride % 2
    vals = np.full(n * stride, np.inf, dtype=np.float32)
    seq = np.zeros(n, np.int32)
    st = np.zeros(n, np.int32)
    for i, (L, off) in enumerate(rows):
        Lp = max(L, 0)
        v = rng.standard_normal(Lp).astype(np.float32)
        if Lp > 10:
            v[rng.integers(0, Lp, size=Lp // 10)] = -0.0
            v[rng.integers(0, Lp, size=Lp // 10)] = 0.0
            v[rng.integers(0, Lp, size=3)] = np.inf
            v[rng.integers(0, Lp, size=3)] = -np.inf
            v[rng.integers(0, Lp, size=5)] = 3e-7  # a binary16 subnormal
        seq[i] = L
        st[i] = off + (i % 3)
        vals[i * stride + st[i]: i * stride + st[i] + Lp] = v
    t = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    half = torch.from_numpy(vals).to(t)
    pages = -(-stride // 16)
    table = rng.choice(1 << 24, size=n * pages, replace=False).astype(np.int32)
    w = wl.Workload("edge", half.to(cuda_device).reshape(n, stride), stride, torch.from_numpy(seq).to(cuda_device),
                    torch.from_numpy(st).to(cuda_device), None, torch.from_numpy(table).to(cuda_device), pages, 16,
                    k, n)
    bits = half.view(torch.int16).numpy().view(np.uint16)
    want = topk_packed_reference(bits, stride, seq, st, None, table, pages, 16, k, dtype=dtype)
    assert np.array_equal(run(w).cpu().numpy(), want)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "long", "mixed"])
def test_bf16_buffer_gives_the_fp32_result_on_bf16_values(cuda_device, name):
    """Every configuration with its scores rounded to bfloat16: the bf16 buffer
    (half the bytes) must give the bits of the fp32 buffer holding the same
    values (the mixed configuration's values are bf16 already), and the
    oracle's result on sampled rows."""
    w32 = wl.named(name, device=cuda_device)
    w16 = wl.with_dtype(w32, "bf16")
    del w32
    w32 = wl.with_dtype(w16, "f32")  # the bf16 values, held as fp32
    out16 = run(w16)
    out32 = run(w32)
    assert torch.equal(out16, out32)
    rows = sample_rows(w16.num_rows, 192)
    want = oracle_rows(w16, rows)
    got = out16[rows.to(out16.device)].cpu().numpy()
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# The register-resident decode kernel (windows of at most 16381 elements):
# each of its three register shapes (4, 8 or 16 elements a thread), tie-heavy
# and sorted values, k from 1 to above the window, every start offset.
# ---------------------------------------------------------------------------
DECODE_CASES = [
    # values, rows, max_len, k, page_size
    ("normal", 24, 4000, 32, 64),      # row stride <= 4093: 4 elements a thread
    ("normal", 24, 8000, 2048, 64),    # <= 8189: 8 elements a thread
    ("normal", 24, 16000, 2048, 64),   # <= 16381: 16 elements a thread
    ("ties", 30, 12000, 777, 1),
    ("bf16", 24, 16000, 2048, 64),
    ("int", 16, 16000, 2048, 16),
    ("equal", 8, 10000, 2048, 64),
    ("ascending", 10, 16000, 2048, 64),
    ("descending", 10, 16000, 300, 64),
    ("normal", 20, 5000, 1, 4),
    ("bf16", 12, 16000, 5000, 64),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=[f"{c[0]}-L{c[2]}-k{c[3]}" for c in DECODE_CASES])
def test_decode_kernel_random_problems(cuda_device, case):
    values, rows, max_len, k, page_size = case
    rng = np.random.default_rng(zlib.crc32(f"decode-{values}-{max_len}-{k}".encode()))
    p = wl.random_problem(rng, rows=rows, max_len=max_len, k=k, page_size=page_size, values=values, slack=13)
    assert p.row_stride <= binding.DECODE_MAX_STRIDE
    w = host_problem_to_device(p, cuda_device)
    before = w.scores.clone()
    want = oracle_host(p)
    assert np.array_equal(run(w, path="decode").cpu().numpy(), want)
    assert np.array_equal(run(w).cpu().numpy(), want), "the automatic choice for short windows"
    assert torch.equal(before, w.scores), "the score buffer was written"


@pytest.mark.parametrize("stride_target", [4093, 8189, 16381])
def test_decode_kernel_edge_lengths_and_offsets(cuda_device, stride_target):
    k = 64
    rng = np.random.default_rng(stride_target)
    lens = [0, 1, k - 1, k, k + 1, 1023, 1024, 1025, 2049, stride_target - 8, -4]
    rows = [(L, off) for L in lens for off in range(4)]
    n = len(rows)
    stride = stride_target if stride_target % 2 else stride_target - 1  # odd
    scores = np.full(n * stride, np.inf, dtype=np.float32)
    seq = np.zeros(n, np.int32)
    st = np.zeros(n, np.int32)
    for i, (L, off) in enumerate(rows):
        Lp = max(L, 0)
        v = rng.standard_normal(Lp).astype(np.float32)
        if Lp > 10:
            v[rng.integers(0, Lp, size=Lp // 10)] = -0.0
            v[rng.integers(0, Lp, size=Lp // 10)] = 0.0
            v[rng.integers(0, Lp, size=3)] = np.inf
            v[rng.integers(0, Lp, size=3)] = -np.inf
        seq[i] = L
        st[i] = min(off + (i % 3), stride - Lp)
        scores[i * stride + st[i]: i * stride + st[i] + Lp] = v
    pages = -(-stride // 16)
    table = rng.choice(1 << 24, size=n * pages, replace=False).astype(np.int32)
    p = wl.HostProblem(scores, stride, seq, st, None, table, pages, 16, k)
    w = host_problem_to_device(p, cuda_device)
    assert np.array_equal(run(w, path="decode").cpu().numpy(), oracle_host(p))


def test_decode_kernel_refuses_long_strides(cuda_device):
    rng = np.random.default_rng(8)
    p = wl.random_problem(rng, rows=4, max_len=binding.DECODE_MAX_STRIDE, k=64, page_size=64, slack=1)
    w = host_problem_to_device(p, cuda_device)
    with pytest.raises(binding.TopkError):
        run(w, path="decode")
    assert np.array_equal(run(w).cpu().numpy(), oracle_host(p))


def test_few_long_rows_full_size(cuda_device):
    """Fewer rows than half the SMs, long windows: the automatic choice splits
    each row over a cluster that merges histograms through distributed shared
    memory; same bits as the split kernel and the oracle's sampled rows."""
    w = wl.few_long(device=cuda_device)
    plan = binding.topk_packed_plan(w.row_stride, w.k, w.num_rows)
    assert plan["path"] == binding.PATHS["stream"] and plan["cluster_size"] > 1
    out = _full_size(w, sample=32)
    assert torch.equal(out, run(w, path="split"))
    w16 = wl.few_long(device=cuda_device, rows=16)
    assert binding.topk_packed_plan(w16.row_stride, w16.k, w16.num_rows)["cluster_size"] == 4
    assert np.array_equal(run(w16).cpu().numpy(), oracle_rows(w16, torch.arange(16)))
