"""The bounds-checked build (libtopk_packed_checked.so, compiled with
TOPK_CHECKED) on the GPU: it stands in for a memory checker.

That build checks, at run time, every global-memory address the kernels
compute (window loads and bulk copies against the row's window rounded out to
16 bytes, page-table reads against the window length, descriptor reads
against num_rows) and every shared-memory index that is not in range by
construction.  A failed check sets bit 2 of the diagnostics word, records its
site in bits 8-15 and skips the access; nothing traps.

The small parity cases of every kernel family run here again through the
checked library: the results must still equal the oracle's, and the
diagnostics word must stay 0.  One case breaks the documented precondition
row_starts[i] + seq_lens[i] <= row_stride inside the allocation (the window
runs into the next buffer row, which is still readable), to show that a
failed check is recorded with its site."""
import zlib

import numpy as np
import pytest
import torch

import tests.test_parity_gpu as tp
from sparse_attention_top_packed_b300 import binding
from sparse_attention_top_packed_b300 import workloads as wl
from tests.gpu_helpers import oracle_rows

pytestmark = pytest.mark.gpu

LAUNCHES = tp.PATHS + [dict(path="decode")]
LAUNCH_IDS = tp.PATH_IDS + ["decode"]


def _serves(launch, stride):
    return launch["path"] != "decode" or stride <= binding.DECODE_MAX_STRIDE


@pytest.fixture(autouse=True)
def _checked_library(cuda_device):
    if not binding.available(checked=True):
        pytest.fail("libtopk_packed_checked.so is not built")
    with binding.checked_build():
        binding.topk_packed_device_flags(reset=True)
        yield
        flags = binding.topk_packed_device_flags(reset=True)
        assert flags == 0, f"diagnostics word {flags:#x}: site {binding.CHECK_SITES.get(binding.check_site(flags))}"


@pytest.mark.parametrize("launch", LAUNCHES, ids=LAUNCH_IDS)
def test_tiny(cuda_device, launch):
    tp.test_tiny(cuda_device, launch)


@pytest.mark.parametrize("launch", tp.PATHS, ids=tp.PATH_IDS)
def test_edge_lengths_and_offsets(cuda_device, launch):
    tp.test_edge_lengths_and_offsets(cuda_device, launch)


CASES = [
    ("normal", 24, 20000, 2048, 64),
    ("ties", 30, 12000, 777, 1),
    ("int", 16, 20000, 2048, 64),
    ("bf16", 50, 3000, 32, 64),
    ("equal", 8, 10000, 2048, 64),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-L{c[2]}-k{c[3]}" for c in CASES])
@pytest.mark.parametrize("launch", LAUNCHES, ids=LAUNCH_IDS)
def test_random_problems(cuda_device, case, launch):
    values, rows, max_len, k, page_size = case
    rng = np.random.default_rng(zlib.crc32(f"checked-{values}-{max_len}-{k}".encode()))
    p = wl.random_problem(rng, rows=rows, max_len=max_len, k=k, page_size=page_size, values=values, slack=13)
    if not _serves(launch, p.row_stride):
        pytest.skip("the decode kernel serves row strides up to TOPK_DECODE_MAX_STRIDE")
    w = tp.host_problem_to_device(p, cuda_device)
    assert np.array_equal(tp.run(w, **launch).cpu().numpy(), tp.oracle_host(p))


@pytest.mark.parametrize("kind", ["falling", "ties", "lengths"])
@pytest.mark.parametrize("path", ["pipe", "split"])
def test_threshold_carried_between_rows(cuda_device, kind, path):
    tp.test_pipe_threshold_carried_between_rows(cuda_device, kind, 1, path)


@pytest.mark.parametrize("launch,case", [(dict(path="split"), 0), (dict(path="multipass"), 0),
                                         (dict(path="decode"), 2)], ids=["split", "multipass", "decode"])
def test_raw_indices_without_page_table(cuda_device, launch, case):
    tp.test_raw_indices_without_page_table(cuda_device, tp.RAW_CASES[case], launch)


def test_large_k(cuda_device):
    tp.test_large_k(cuda_device, 4096)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_half_width(cuda_device, dtype):
    tp.test_half_width_random_problems(cuda_device, dtype, "normal", 24, 20000, 2048)
    tp.test_half_width_edge_lengths_offsets_and_specials(cuda_device, dtype)


def test_prefill_rows_on_the_automatic_path(cuda_device):
    """The first 296 rows of the ISL-70000 prefill batch (two per SM), as the
    benchmark launches them: sampled thresholds, carried hints and the staged
    page rows of the split kernel."""
    w = wl.named("prefill", device=cuda_device).head(296)
    out = torch.empty((w.num_rows, w.k), dtype=torch.int32, device=cuda_device)
    binding.topk_packed(w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch, w.page_table,
                        w.pt_stride, w.page_size, w.k, out, w.num_rows)
    torch.cuda.synchronize()
    rows = torch.arange(0, w.num_rows, 7)
    assert np.array_equal(out[rows].cpu().numpy(), oracle_rows(w, rows))


@pytest.mark.parametrize("launch", LAUNCHES, ids=LAUNCH_IDS)
def test_a_window_past_its_row_is_recorded(cuda_device, launch):
    """Row 1's window runs 700 elements into row 2 of the buffer (a broken
    precondition; the memory is still inside the allocation).  The checked
    build records site 1 and still reads the row, so the result is the
    oracle's reading of the flat buffer."""
    rng = np.random.default_rng(11)
    rows, stride, k = 4, 6000, 512
    scores = rng.standard_normal(rows * stride).astype(np.float32)
    seq = np.array([5000, 3000, 4000, 100], np.int32)
    st = np.array([0, stride - 2300, 1000, 7], np.int32)
    pages = -(-(stride + 1000) // 16)
    table = rng.choice(1 << 24, size=rows * pages, replace=False).astype(np.int32)
    p = wl.HostProblem(scores, stride, seq, st, None, table, pages, 16, k)
    w = tp.host_problem_to_device(p, cuda_device)
    out = tp.run(w, **launch)
    flags = binding.topk_packed_device_flags(reset=True)
    assert flags & binding.FLAG_OUT_OF_BOUNDS, f"{flags:#x}"
    assert binding.check_site(flags) == 1, binding.CHECK_SITES.get(binding.check_site(flags))
    assert flags & (binding.FLAG_STREAM_WAIT_TIMEOUT | binding.FLAG_BAD_OUTPUT_POSITION) == 0
    assert np.array_equal(out.cpu().numpy(), tp.oracle_host(p))
