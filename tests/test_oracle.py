"""Pins of the CPU oracle (no GPU).

The oracle (oracle/topk_oracle.c) is checked against things other than itself:
  * hand-worked examples (tests/golden/page_transform_example.json);
  * the closed-form rank of each element (oracle/brute_force.py), on >= 10^4
    random tiny rows with heavy ties, signed zeros and infinities;
  * special cases that reduce to a library routine (k >= L: the identity
    selection; page_size 1 with an identity table: raw indices; numpy lexsort);
  * the invariants of oracle/invariants.py on larger rows;
  * metamorphic relations that follow from the definition: exact power-of-two
    scaling, values outside the windows, a permuted page table with the row
    map following it, reversed windows;
  * planted mistakes: mutated copies of the oracle source must fail these pins.
"""
import dataclasses
import json
import os

import numpy as np
import pytest

from oracle import topk_packed_reference
from oracle import brute_force
from oracle.invariants import InvariantError, check_row
from sparse_attention_top_packed_b300.workloads import random_problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_transform_example.json")


def _f(x):
    return float(x)


def run_oracle(p, **kw):
    return topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch,
                                 p.page_table, p.pt_stride, p.page_size, p.k, **kw)


def test_golden_examples():
    data = json.load(open(GOLDEN))
    for ex in data["examples"]:
        values = np.array([_f(v) for v in ex["values"]], dtype=np.float32)
        for case in ex["cases"]:
            k = case["k"]
            got = topk_packed_reference(values, 0, [len(values)], [0], None,
                                        np.array(ex["page_row"]), 0, ex["page_size"], k)
            assert got[0].tolist() == case["expected"], (ex["name"], k)
            # the same row placed at an unaligned offset inside a row of +inf
            stride = len(values) + 11
            buf = np.full(2 * stride, np.inf, dtype=np.float32)
            buf[stride + 3: stride + 3 + len(values)] = values
            got2 = topk_packed_reference(buf, stride, [0, len(values)], [0, 3], [0, 0],
                                         np.array(ex["page_row"]), 0, ex["page_size"], k)
            assert got2[1].tolist() == case["expected"], (ex["name"], k, "offset")
            assert got2[0].tolist() == [-1] * k
            # and the brute force agrees with the fixture too
            assert brute_force.row_result(values.tolist(), ex["page_row"], ex["page_size"], k) \
                == case["expected"]


def _brute_rows(p):
    return brute_force.packed_result(p.scores, p.row_stride, p.seq_lens, p.row_starts,
                                     p.row_to_batch, p.page_table, p.pt_stride, p.page_size, p.k)


@pytest.mark.parametrize("values", ["ties", "normal", "int", "equal", "bf16"])
def test_oracle_matches_pure_python_rank(values):
    rng = np.random.default_rng(1234 + len(values))
    for trial in range(20):
        k = int(rng.integers(1, 40))
        p = random_problem(rng, rows=12, max_len=int(rng.integers(1, 48)), k=k,
                           page_size=int(rng.choice([1, 2, 4, 16])), values=values,
                           identity=bool(trial % 3 == 0))
        assert run_oracle(p).tolist() == _brute_rows(p), (values, trial)


def test_oracle_matches_rank_on_ten_thousand_tiny_rows():
    """>= 10^4 rows, n <= 64, k <= n + 8, tie-heavy values including +-0 and +-inf."""
    rng = np.random.default_rng(7)
    rows_checked = 0
    while rows_checked < 10240:
        kind = ["ties", "int", "normal", "bf16"][rows_checked // 256 % 4]
        max_len = int(rng.integers(1, 65))
        k = int(rng.integers(1, max_len + 9))
        p = random_problem(rng, rows=64, max_len=max_len, k=k,
                           page_size=int(rng.choice([1, 4, 64])), values=kind)
        got = run_oracle(p)
        for i in range(p.num_rows):
            L = int(p.seq_lens[i])
            base = i * p.row_stride + int(p.row_starts[i])
            chosen = brute_force.select_by_rank_np(p.scores[base: base + L], k)
            b = int(p.row_to_batch[i])
            page_row = p.page_table[b * p.pt_stride:(b + 1) * p.pt_stride]
            expect = [brute_force.page_slot(page_row, p.page_size, int(j)) for j in chosen]
            expect += [-1] * (k - len(expect))
            assert got[i].tolist() == expect, (kind, rows_checked + i)
        rows_checked += p.num_rows


def test_oracle_matches_rank_for_k_above_2048():
    """k of 2049, 4096 and 5000 on windows of up to 6000 (so the selection is
    neither trivial nor the whole window), against the closed-form rank."""
    rng = np.random.default_rng(2049)
    for k, values in [(2049, "normal"), (4096, "bf16"), (5000, "int")]:
        p = random_problem(rng, rows=4, max_len=6000, k=k, page_size=64, values=values,
                           forced_lens=[6000, 5999, k + 1, k - 1])
        got = run_oracle(p)
        for i in range(p.num_rows):
            L = int(p.seq_lens[i])
            base = i * p.row_stride + int(p.row_starts[i])
            chosen = brute_force.select_by_rank_np(p.scores[base: base + L], k)
            b = int(p.row_to_batch[i])
            page_row = p.page_table[b * p.pt_stride:(b + 1) * p.pt_stride]
            expect = [brute_force.page_slot(page_row, p.page_size, int(j)) for j in chosen]
            expect += [-1] * (k - len(expect))
            assert got[i].tolist() == expect, (k, values, i)


def test_k_at_least_window_is_identity_selection():
    rng = np.random.default_rng(3)
    p = random_problem(rng, rows=30, max_len=200, k=256, page_size=16, values="normal")
    got = run_oracle(p)
    for i in range(p.num_rows):
        L = int(p.seq_lens[i])
        b = int(p.row_to_batch[i])
        j = np.arange(L)
        pages = p.page_table[b * p.pt_stride + (j // 16)]
        expect = np.concatenate([pages.astype(np.int64) * 16 + j % 16, -np.ones(256 - L)])
        assert np.array_equal(got[i], expect.astype(np.int32))


def test_unit_pages_identity_table_gives_raw_indices_and_matches_lexsort():
    rng = np.random.default_rng(5)
    rows, L, k = 40, 500, 37
    p = random_problem(rng, rows=rows, max_len=L, k=k, page_size=1, values="bf16",
                       forced_lens=[L] * rows)
    table = np.tile(np.arange(p.pt_stride, dtype=np.int32), rows)
    got = topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts,
                                np.arange(rows), table, p.pt_stride, 1, k)
    for i in range(rows):
        base = i * p.row_stride + int(p.row_starts[i])
        w = p.scores[base: base + L].astype(np.float64)
        order = np.lexsort((np.arange(L), -w))  # primary: -w ascending, then index
        assert got[i].tolist() == sorted(order[:k].tolist())


def test_raw_indices_without_a_page_table_match_the_rank_definition():
    """page_table None: the selected window indices themselves, ascending, then
    -1; checked against the closed-form rank on tie-heavy tiny rows."""
    rng = np.random.default_rng(21)
    for trial in range(60):
        kind = ["ties", "int", "normal", "bf16", "equal"][trial % 5]
        max_len = int(rng.integers(1, 65))
        k = int(rng.integers(1, max_len + 9))
        p = random_problem(rng, rows=16, max_len=max_len, k=k, page_size=4, values=kind)
        got = topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch,
                                    None, 0, 4, k)
        for i in range(p.num_rows):
            L = int(p.seq_lens[i])
            base = i * p.row_stride + int(p.row_starts[i])
            chosen = brute_force.select_by_rank_np(p.scores[base: base + L], k)
            expect = [int(j) for j in chosen] + [-1] * (k - len(chosen))
            assert got[i].tolist() == expect, (kind, trial, i)
        assert got.tolist() == brute_force.packed_result(p.scores, p.row_stride, p.seq_lens, p.row_starts,
                                                         p.row_to_batch, None, 0, 4, k)


def test_raw_indices_equal_unit_pages_through_an_identity_table():
    rng = np.random.default_rng(23)
    p = random_problem(rng, rows=20, max_len=400, k=50, page_size=1, values="ties")
    table = np.tile(np.arange(p.pt_stride, dtype=np.int32), p.num_rows)
    via_table = topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts,
                                      np.arange(p.num_rows), table, p.pt_stride, 1, 50)
    raw = topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch,
                                None, 0, 1, 50)
    assert np.array_equal(raw, via_table)


def test_invariants_hold_on_larger_rows():
    rng = np.random.default_rng(11)
    for values in ["normal", "bf16", "int", "ties"]:
        p = random_problem(rng, rows=16, max_len=5000, k=300, page_size=64, values=values)
        got = run_oracle(p)
        for i in range(p.num_rows):
            L = int(p.seq_lens[i])
            base = i * p.row_stride + int(p.row_starts[i])
            b = int(p.row_to_batch[i])
            check_row(p.scores[base: base + L], p.page_table[b * p.pt_stride:(b + 1) * p.pt_stride],
                      p.page_size, p.k, got[i])


def test_invariant_checker_catches_planted_errors():
    v = np.array([0.5, 2.0, -1.0, 2.0, 0.5, 3.0], dtype=np.float32)
    pages = [7, 2]
    check_row(v, pages, 4, 4, [28, 29, 31, 9])
    bad = {
        "tie to higher index": [29, 31, 8, 9],
        "not ascending": [29, 28, 31, 9],
        "foreign page": [28, 29, 31, 41],
        "too few": [28, 29, 31, -1],
        "lower score chosen": [28, 29, 30, 9],
    }
    for name, out in bad.items():
        with pytest.raises(InvariantError):
            check_row(v, pages, 4, 4, out)
            pytest.fail(name)


def test_oracle_rejects_bad_arguments():
    for kw in [dict(k=0), dict(page_size=3), dict(page_size=0)]:
        args = dict(k=2, page_size=4)
        args.update(kw)
        with pytest.raises(ValueError):
            topk_packed_reference(np.zeros(4, np.float32), 4, [4], [0], None, np.zeros(4),
                                  0, args["page_size"], args["k"])
    # without a page table the page size is not used
    out = topk_packed_reference(np.array([1, 3, 2, 0], np.float32), 4, [4], [0], None, None, -1, 3, 2)
    assert out.tolist() == [[1, 2]]


def test_oracle_thread_count_does_not_change_result():
    rng = np.random.default_rng(9)
    p = random_problem(rng, rows=50, max_len=3000, k=100, page_size=64, values="bf16")
    a = run_oracle(p, nthreads=1)
    b = run_oracle(p, nthreads=7)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# Metamorphic pins: transformations of the input whose effect on the result
# follows from the definition alone.
# ---------------------------------------------------------------------------
def _windows_mask(p):
    """True at every cell of `scores` that lies inside some row's window."""
    inside = np.zeros(p.scores.shape[0], dtype=bool)
    for i in range(p.num_rows):
        L = max(int(p.seq_lens[i]), 0)
        base = i * p.row_stride + int(p.row_starts[i])
        inside[base: base + L] = True
    return inside


@pytest.mark.parametrize("values", ["normal", "ties", "bf16", "int"])
def test_exact_power_of_two_scaling_keeps_the_result(values):
    """Scaling every score by 2^e (exact in float32 for these magnitudes)
    keeps every comparison, so the result is unchanged; -0.0 stays equal to
    +0.0 and the infinities stay infinite."""
    rng = np.random.default_rng(31)
    p = random_problem(rng, rows=20, max_len=300, k=40, page_size=8, values=values)
    base = run_oracle(p)
    for e in (-3, 5):
        q = dataclasses.replace(p, scores=(p.scores * np.float32(2.0 ** e)).astype(np.float32))
        assert np.array_equal(run_oracle(q), base), e


def test_values_outside_the_windows_do_not_matter():
    rng = np.random.default_rng(33)
    p = random_problem(rng, rows=24, max_len=500, k=64, page_size=16, values="ties")
    base = run_oracle(p)
    inside = _windows_mask(p)
    for fill in (np.float32(np.inf), np.float32(-np.inf), np.float32(1e30)):
        s = p.scores.copy()
        s[~inside] = fill
        assert np.array_equal(run_oracle(dataclasses.replace(p, scores=s)), base)
    s = p.scores.copy()
    s[~inside] = rng.standard_normal(int((~inside).sum())).astype(np.float32) * 100
    assert np.array_equal(run_oracle(dataclasses.replace(p, scores=s)), base)


def test_page_table_rows_follow_the_row_map():
    """Permuting the page table's rows and the row map with it leaves every
    output unchanged: a row reads its pages only through row_to_batch."""
    rng = np.random.default_rng(35)
    p = random_problem(rng, rows=30, max_len=400, k=50, page_size=16, values="normal", table_rows=6)
    base = run_oracle(p)
    n_table = p.page_table.size // p.pt_stride
    perm = rng.permutation(n_table)
    table = p.page_table.reshape(n_table, p.pt_stride)
    moved = np.empty_like(table)
    moved[perm] = table  # old row b now sits at perm[b]
    rtb = perm[p.row_to_batch].astype(np.int32)
    q = dataclasses.replace(p, page_table=moved.reshape(-1), row_to_batch=rtb)
    assert np.array_equal(run_oracle(q), base)


def test_reversed_windows_mirror_the_selection_up_to_ties():
    """On tie-free rows, reversing each window maps index j to L-1-j, so the
    selected set is mirrored (raw indices, no page table)."""
    rng = np.random.default_rng(37)
    p = random_problem(rng, rows=16, max_len=300, k=30, page_size=1, values="normal")
    raw = topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts, None, None, 0, 1, 30)
    s = p.scores.copy()
    for i in range(p.num_rows):
        L = max(int(p.seq_lens[i]), 0)
        base = i * p.row_stride + int(p.row_starts[i])
        s[base: base + L] = s[base: base + L][::-1]
    rev = topk_packed_reference(s, p.row_stride, p.seq_lens, p.row_starts, None, None, 0, 1, 30)
    for i in range(p.num_rows):
        L = max(int(p.seq_lens[i]), 0)
        m = min(L, 30)
        want = sorted(L - 1 - int(j) for j in raw[i, :m])
        assert rev[i, :m].tolist() == want and (rev[i, m:] == -1).all()


# ---------------------------------------------------------------------------
# 16-bit score buffers (bfloat16, IEEE binary16): the oracle turns each element
# into its exact value first.  Pinned by hand-encoded examples, by the
# libraries' own decoders (numpy float16, torch bfloat16) and by the
# closed-form rank on tie-heavy rows with special values.
# ---------------------------------------------------------------------------
HALF_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "half_width_example.json")


def test_half_width_golden_examples():
    data = json.load(open(HALF_GOLDEN))
    checked = 0
    for ex in data["examples"]:
        for dtype in ("bf16", "f16"):
            if dtype not in ex:
                continue
            bits = np.array([int(h, 16) for h in ex[dtype]], dtype=np.uint16)
            for case in ex["cases"]:
                got = topk_packed_reference(bits, 0, [len(bits)], [0], None, np.array(ex["page_row"], np.int32),
                                            0, ex["page_size"], case["k"], dtype=dtype)
                assert got[0].tolist() == case["expected"], (ex["name"], dtype, case)
                checked += 1
    assert checked >= 10


def _half_problem(rng, dtype, rows=16, max_len=300, k=None):
    """Random 16-bit patterns (no NaN) in ragged windows; cells outside the
    windows hold the pattern of +inf."""
    stride = max_len + 5
    inf = 0x7C00 if dtype == "f16" else 0x7F80
    bits = np.full(rows * stride, inf, dtype=np.uint16)
    seq = rng.integers(0, max_len + 1, size=rows).astype(np.int32)
    starts = np.array([rng.integers(0, stride - L + 1) for L in seq], dtype=np.int32)
    for i in range(rows):
        L = int(seq[i])
        b = rng.integers(0, 1 << 16, size=L).astype(np.uint16)
        # NaN patterns (exponent all ones, fraction non-zero) become the
        # infinity of the same sign: NaN is outside the contract
        frac = 0x03FF if dtype == "f16" else 0x007F
        nan = ((b & (0x7FFF ^ frac)) == (0x7FFF ^ frac)) & ((b & frac) != 0)
        b[nan] &= np.uint16(0xFFFF ^ frac)
        # a few repeated values to make ties
        if L > 4:
            b[rng.integers(0, L, size=L // 4)] = b[rng.integers(0, L)]
        bits[i * stride + starts[i]: i * stride + starts[i] + L] = b
    table = rng.choice(1 << 20, size=4 * (-(-stride // 16)), replace=False).astype(np.int32)
    rtb = rng.integers(0, 4, size=rows).astype(np.int32)
    kk = int(k if k is not None else rng.integers(1, max_len))
    return bits, stride, seq, starts, rtb, table, -(-stride // 16), 16, kk


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_f16_buffer_equals_numpy_float16_values(seed):
    """numpy's float16 decoder (a library routine) against the oracle's own."""
    rng = np.random.default_rng(seed)
    bits, stride, seq, starts, rtb, table, pts, ps, k = _half_problem(rng, "f16")
    as_f32 = bits.view(np.float16).astype(np.float32)
    a = topk_packed_reference(bits, stride, seq, starts, rtb, table, pts, ps, k, dtype="f16")
    b = topk_packed_reference(as_f32, stride, seq, starts, rtb, table, pts, ps, k)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("seed", [4, 5, 6])
def test_bf16_buffer_equals_torch_bfloat16_values(seed):
    """torch's bfloat16 decoder (a library routine) against the oracle's own."""
    import torch

    rng = np.random.default_rng(seed)
    bits, stride, seq, starts, rtb, table, pts, ps, k = _half_problem(rng, "bf16")
    as_f32 = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    a = topk_packed_reference(bits, stride, seq, starts, rtb, table, pts, ps, k, dtype="bf16")
    b = topk_packed_reference(as_f32, stride, seq, starts, rtb, table, pts, ps, k)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_half_width_oracle_matches_rank(dtype):
    """The closed-form rank on rows of 16-bit values drawn from a tie-heavy set
    with signed zeros, infinities, subnormals and the extremes (values decoded
    by the libraries), against the oracle reading the bit patterns."""
    import torch

    if dtype == "f16":
        pool = np.array([0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0xBC00, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00,
                         0x3C01], dtype=np.uint16)
        decode = lambda b: b.view(np.float16).astype(np.float64)
    else:
        pool = np.array([0x0000, 0x8000, 0x0001, 0x007F, 0x0080, 0x3F80, 0xBF80, 0x7F7F, 0xFF7F, 0x7F80, 0xFF80,
                         0x3F81], dtype=np.uint16)
        decode = lambda b: torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    rng = np.random.default_rng(99)
    for trial in range(200):
        n = int(rng.integers(0, 40))
        k = int(rng.integers(1, 44))
        b = pool[rng.integers(0, pool.shape[0], size=n)]
        got = topk_packed_reference(b, 0, [n], [0], None, None, 0, 1, k, dtype=dtype)[0].tolist()
        chosen = brute_force.select_by_rank_np(decode(b), k).tolist()
        assert got == chosen + [-1] * (k - len(chosen)), (dtype, trial)
