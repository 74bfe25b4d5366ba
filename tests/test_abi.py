"""The C ABI on the host (no GPU): the library loads, exports every function
include/topk_packed.h declares, and rejects bad arguments with the documented
status before touching the device."""
import ctypes
import os
import re

import pytest

from sparse_attention_top_packed_b300 import binding
from sparse_attention_top_packed_b300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "topk_packed.h")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return ctypes.CDLL(binding.library_path())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(topk_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["topk_packed", "topk_packed_ex", "topk_packed_plan", "topk_status_string",
              "topk_last_cuda_error", "topk_packed_device_flags"]:
        assert n in names


def test_library_exports_every_declared_function(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_exports_nothing_else(lib):
    out = os.popen(f"nm -D --defined-only {binding.library_path()}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions())


def test_checked_library_exports_the_same_functions(lib):
    """The bounds-checked build is the same ABI."""
    path = binding.library_path(checked=True)
    assert os.path.exists(path)
    checked = ctypes.CDLL(path)
    assert all(hasattr(checked, n) for n in declared_functions())
    out = os.popen(f"nm -D --defined-only {path}").read()
    assert {line.split()[-1] for line in out.splitlines() if " T " in line} == set(declared_functions())
    with binding.checked_build():
        assert binding.library_path() == path
        assert binding.topk_status_string(0)
    assert binding.library_path() != path


def test_check_site_field():
    assert binding.check_site(binding.FLAG_OUT_OF_BOUNDS | (5 << 8)) == 5
    assert binding.check_site(binding.FLAG_STREAM_WAIT_TIMEOUT) == 0
    assert set(binding.CHECK_SITES) == set(range(1, 11))


def test_status_strings(lib):
    for code, name in binding.STATUS_NAMES.items():
        assert binding.topk_status_string(code)
    assert binding.topk_status_string(99) == "unknown status"


def _call(k=8, page_size=64, num_rows=1, row_stride=16, pt_stride=1, scores=0x1000,
          seq=0x2000, starts=0x3000, rtb=None, table=0x4000, out=0x5000, cfg=None):
    args = [scores, row_stride, seq, starts, rtb, table, pt_stride, page_size, k, out, num_rows]
    if cfg is None:
        return binding.raw_call("topk_packed", *args, None)
    return binding.raw_call("topk_packed_ex", *args, ctypes.byref(cfg), None)


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    INVALID, UNSUPPORTED, OK = 1, 2, 0
    assert _call(k=0) == INVALID
    assert _call(k=-3) == INVALID
    assert _call(page_size=0) == INVALID
    assert _call(page_size=48) == INVALID
    assert _call(num_rows=-1) == INVALID
    assert _call(row_stride=-1) == INVALID
    assert _call(pt_stride=-5) == INVALID
    assert _call(scores=None) == INVALID
    assert _call(seq=None) == INVALID
    assert _call(starts=None) == INVALID
    assert _call(out=None) == INVALID
    assert _call(k=(1 << 20) + 1) == UNSUPPORTED
    assert _call(scores=0x1002) == UNSUPPORTED  # not 4-byte aligned
    # nothing to do: success without a device
    assert _call(num_rows=0, scores=None, seq=None, starts=None, table=None, out=None) == OK
    bad = binding.LaunchConfig(7, 0, 0)
    assert _call(cfg=bad) == INVALID
    bad = binding.LaunchConfig(6, 0, 0)
    assert _call(cfg=bad) == INVALID
    dec = binding.LaunchConfig(5, 0, 0)  # the decode kernel: accepted; the next check answers
    assert _call(cfg=dec, scores=0x1002) == UNSUPPORTED
    bad = binding.LaunchConfig(2, 3, 0)
    assert _call(cfg=bad) == INVALID
    bad = binding.LaunchConfig(2, 0, -1)
    assert _call(cfg=bad) == INVALID
    bad = binding.LaunchConfig(3, 0, 0, 0, 2)  # an unknown test flag
    assert _call(cfg=bad) == INVALID
    bad = binding.LaunchConfig(3, 0, 0, 0, 0, 2)  # dependent_launch is 0 or 1
    assert _call(cfg=bad) == INVALID
    dep = binding.LaunchConfig(4, 0, 0, 0, 0, 1)
    assert _call(cfg=dep, scores=0x1002) == UNSUPPORTED  # accepted; the next check answers
    known = binding.LaunchConfig(3, 0, 0, 1000, binding.TEST_UNSATISFIED_WAIT)
    assert _call(cfg=known, scores=0x1002) == UNSUPPORTED  # accepted; the next check answers


def test_null_page_table_means_raw_indices_and_frees_page_arguments(lib):
    """Without a page table the output is the window index itself, so
    page_size and pt_stride are not checked.  Every call here stops at a
    later check, before any device work (the pointers are not real)."""
    INVALID, UNSUPPORTED, OK = 1, 2, 0
    # a NULL table passes the pointer checks: the next check (alignment) answers
    assert _call(table=None, scores=0x1002) == UNSUPPORTED
    # page_size and pt_stride are ignored without a table, checked with one
    assert _call(table=None, page_size=48, pt_stride=-5, k=(1 << 20) + 1) == UNSUPPORTED
    assert _call(page_size=48, k=(1 << 20) + 1) == INVALID
    assert _call(pt_stride=-5, k=(1 << 20) + 1) == INVALID
    assert _call(table=None, num_rows=0, page_size=0) == OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_libs", {})
    monkeypatch.setattr(binding, "library_path", lambda checked=None: str(tmp_path / "missing.so"))
    with pytest.raises(binding.TopkError):
        binding.topk_status_string(0)


def _typed(dtype, scores=0x1000, k=8, cfg=None):
    args = [scores, dtype, 16, 0x2000, 0x3000, None, 0x4000, 1, 64, k, 0x5000, 1]
    return binding.raw_call("topk_packed_typed", *args, None if cfg is None else ctypes.byref(cfg), None)


def test_typed_entry_point_checks(lib):
    INVALID, UNSUPPORTED = 1, 2
    assert _typed(3) == INVALID  # unknown element type
    assert _typed(-1) == INVALID
    assert _typed(1, scores=0x1001) == UNSUPPORTED  # bf16 needs 2-byte alignment
    assert _typed(2, k=2049) == UNSUPPORTED         # 16-bit buffers: k <= TOPK_K_FAST
    for path in (1, 2, 3):                           # 16-bit buffers: split kernel only
        assert _typed(1, cfg=binding.LaunchConfig(path, 0, 0)) == UNSUPPORTED
    assert _typed(0, scores=0x1002) == UNSUPPORTED  # f32 needs 4-byte alignment
