"""Planted mistakes: each mutated copy of the C oracle must fail the pins.

A mutant is the oracle source with one plausible mistake written in (a wrong
sign, a flipped tie rule, a dropped term, a transposed operand, ...), compiled
into a temporary library on the CPU.  The pins of test_oracle.py -- the
hand-worked examples and the closed-form rank -- must reject every mutant,
which shows they are strong enough to catch such a mistake in the oracle.
"""
import ctypes
import json
import os

import numpy as np
import pytest

from oracle import build as oracle_build
from oracle import brute_force
from sparse_attention_top_packed_b300.workloads import random_problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_transform_example.json")

MUTANTS = {
    "tie to higher index": ("return (a->j > b->j) - (a->j < b->j);",
                            "return (a->j < b->j) - (a->j > b->j);"),
    "k smallest instead of largest": ("if (a->v > b->v) return -1;\n  if (a->v < b->v) return 1;",
                                      "if (a->v > b->v) return 1;\n  if (a->v < b->v) return -1;"),
    "output left in rank order": ("qsort(chosen, (size_t)m, sizeof(int32_t), by_index_asc);", ";"),
    "window offset dropped": ("(int64_t)i * p->row_stride + p->row_starts[i];",
                              "(int64_t)i * p->row_stride;"),
    "table-row map ignored": ("p->row_to_batch ? (int64_t)p->row_to_batch[i] : (int64_t)i;",
                              "(int64_t)i;"),
    "page and offset transposed": (
        "page_row[j >> page_bits] * p->page_size + (j & (p->page_size - 1))",
        "page_row[j & (p->page_size - 1)] * p->page_size + (j >> page_bits)"),
    "offset mask off by one": ("(j & (p->page_size - 1))", "(j & p->page_size)"),
    "table stride dropped": ("table_row * p->pt_stride", "table_row"),
    "padding with zero": ("out_row[t] = -1;", "out_row[t] = 0;"),
    "one slot short": ("const int32_t m = n < p->k ? n : p->k;",
                       "const int32_t m = n < p->k ? n : p->k - 1;"),
    "raw index off by one": ("for (int32_t t = 0; t < m; ++t) out_row[t] = chosen[t];",
                             "for (int32_t t = 0; t < m; ++t) out_row[t] = chosen[t] + 1;"),
    "raw rows left unpadded": ("if (p->page_table == NULL) {\n    for (int32_t t = 0; t < m; ++t) out_row[t] = chosen[t];\n  }",
                               "if (p->page_table == NULL) {\n    for (int32_t t = 0; t < m; ++t) out_row[t] = chosen[t];\n    return;\n  }"),
}


# planted mistakes in the decoding of 16-bit buffers (each changes the order
# of some values, so a correct pin must notice)
HALF_MUTANTS = {
    "binary16 subnormals decoded as normals": ("if (e == 0)\n    mag = ldexpf((float)m, -24);\n  else if",
                                               "if (0)\n    mag = ldexpf((float)m, -24);\n  else if"),
    "binary16 exponent field misread": ("e = (h >> 10) & 31", "e = (h >> 11) & 31"),
    "bfloat16 pattern shifted one bit short": ("(uint32_t)h << 16", "(uint32_t)h << 15"),
}
HALF_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "half_width_example.json")


def _compile(tmp_path, name, find, replace):
    src = open(oracle_build.SOURCE).read()
    assert src.count(find) == 1, f"mutation site for {name!r} not found exactly once"
    path = tmp_path / (name.replace(" ", "_") + ".c")
    path.write_text(src.replace(find, replace))
    lib_path = str(tmp_path / (name.replace(" ", "_") + ".so"))
    oracle_build.build(str(path), lib_path, extra_flags=("-w",))
    lib = ctypes.CDLL(lib_path)
    lib.topk_oracle_typed.restype = ctypes.c_int
    lib.topk_oracle_typed.argtypes = [
        ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
        ctypes.c_int32, ctypes.c_int32]
    lib.topk_oracle.restype = ctypes.c_int
    lib.topk_oracle.argtypes = [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
        ctypes.c_int32, ctypes.c_int32]
    return lib


def _call(lib, scores, row_stride, seq_lens, row_starts, rtb, table, pt_stride, page_size, k):
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    rs = np.ascontiguousarray(row_starts, dtype=np.int32)
    rb = None if rtb is None else np.ascontiguousarray(rtb, dtype=np.int32)
    pt = None if table is None else np.ascontiguousarray(table, dtype=np.int32)
    out = np.full((sl.shape[0], k), 12345, dtype=np.int32)
    lib.topk_oracle(sc.ctypes.data, row_stride, sl.ctypes.data, rs.ctypes.data,
                    None if rb is None else rb.ctypes.data, None if pt is None else pt.ctypes.data,
                    pt_stride, page_size, k, out.ctypes.data, sl.shape[0], 1)
    return out


def _passes_pins(lib) -> bool:
    data = json.load(open(GOLDEN))
    for ex in data["examples"]:
        values = np.array([float(v) for v in ex["values"]], dtype=np.float32)
        for case in ex["cases"]:
            got = _call(lib, values, 0, [len(values)], [0], None, np.array(ex["page_row"]), 0,
                        ex["page_size"], case["k"])
            if got[0].tolist() != case["expected"]:
                return False
    rng = np.random.default_rng(42)
    for trial in range(24):
        p = random_problem(rng, rows=8, max_len=40, k=int(rng.integers(1, 30)),
                           page_size=[1, 4, 16][trial % 3], values=["ties", "normal"][trial % 2],
                           identity=trial % 4 == 0)
        got = _call(lib, p.scores, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch,
                    p.page_table, p.pt_stride, p.page_size, p.k)
        want = brute_force.packed_result(p.scores, p.row_stride, p.seq_lens, p.row_starts,
                                         p.row_to_batch, p.page_table, p.pt_stride, p.page_size,
                                         p.k)
        if got.tolist() != want:
            return False
        # and without a page table: raw window indices
        got = _call(lib, p.scores, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch,
                    None, 0, p.page_size, p.k)
        want = brute_force.packed_result(p.scores, p.row_stride, p.seq_lens, p.row_starts,
                                         p.row_to_batch, None, 0, p.page_size, p.k)
        if got.tolist() != want:
            return False
    return True


def test_unmutated_source_passes(tmp_path):
    lib = _compile(tmp_path, "clean", "int topk_oracle(", "int topk_oracle(")
    assert _passes_pins(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    find, replace = MUTANTS[name]
    lib = _compile(tmp_path, name, find, replace)
    assert not _passes_pins(lib), f"pins did not catch the planted mistake: {name}"


def _passes_half_pins(lib) -> bool:
    """The 16-bit pins of test_oracle.py: the hand-encoded examples and the
    libraries' decoders."""
    import torch

    def call(bits, dtype, page_row, page_size, k):
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        pt = np.ascontiguousarray(page_row, dtype=np.int32)
        sl = np.array([b.shape[0]], np.int32)
        rs = np.zeros(1, np.int32)
        out = np.full((1, k), 12345, dtype=np.int32)
        lib.topk_oracle_typed(b.ctypes.data, {"bf16": 1, "f16": 2}[dtype], 0, sl.ctypes.data, rs.ctypes.data, None,
                              pt.ctypes.data, 0, page_size, k, out.ctypes.data, 1, 1)
        return out[0].tolist()

    data = json.load(open(HALF_GOLDEN))
    for ex in data["examples"]:
        for dtype in ("bf16", "f16"):
            if dtype in ex:
                bits = [int(h, 16) for h in ex[dtype]]
                for case in ex["cases"]:
                    if call(bits, dtype, ex["page_row"], ex["page_size"], case["k"]) != case["expected"]:
                        return False
    rng = np.random.default_rng(5)
    for dtype in ("f16", "bf16"):
        for _ in range(20):
            n = int(rng.integers(1, 60))
            b = rng.integers(0, 1 << 16, size=n).astype(np.uint16)
            if dtype == "f16":
                b = b[((b >> 10) & 31) != 31]
                vals = b.view(np.float16).astype(np.float64)
            else:
                b = b[((b >> 7) & 255) != 255]
                vals = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
            k = int(rng.integers(1, n + 2))
            want = brute_force.select_by_rank_np(vals, k).tolist()
            want = want + [-1] * (k - len(want))
            if call(b, dtype, np.arange(max(len(b), 1)), 1, k) != want:
                return False
    return True


def test_unmutated_source_passes_half_width_pins(tmp_path):
    lib = _compile(tmp_path, "clean_half", "int topk_oracle_typed(", "int topk_oracle_typed(")
    assert _passes_half_pins(lib)


@pytest.mark.parametrize("name", sorted(HALF_MUTANTS))
def test_half_width_mutant_is_caught(tmp_path, name):
    find, replace = HALF_MUTANTS[name]
    lib = _compile(tmp_path, name, find, replace)
    assert not _passes_half_pins(lib), f"pins did not catch the planted mistake: {name}"
