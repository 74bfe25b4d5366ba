"""ctypes binding of libtopk_packed.so (argument marshalling only).

Every function has the name and argument order of its C counterpart in
``include/topk_packed.h``.  Tensors are passed as their device pointers; the
C library validates sizes and launches the CUDA kernels.  There is no
fallback: if the shared library is missing or the device is not sm_103a the
call raises.

``checked_build()`` routes the calls made inside it to
libtopk_packed_checked.so, the same library compiled with run-time bounds
checks (a failed check sets bit 2 of the diagnostics word and records its
site in bits 8-15); it is for testing, not for speed.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libtopk_packed.so"
CHECKED_LIB_NAME = "libtopk_packed_checked.so"

TOPK_OK = 0
STATUS_NAMES = {0: "TOPK_OK", 1: "TOPK_ERR_INVALID_ARG", 2: "TOPK_ERR_UNSUPPORTED",
                3: "TOPK_ERR_LAUNCH", 4: "TOPK_ERR_DEVICE"}
PATHS = {"auto": 0, "multipass": 1, "stream": 2, "pipe": 3, "split": 4, "decode": 5}
DECODE_MAX_STRIDE = 16381
K_MAX = 1 << 20
K_FAST = 2048


class TopkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class LaunchConfig(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("cluster_size", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("stream_wait_ns", ctypes.c_uint32),
                ("test_flags", ctypes.c_uint32), ("dependent_launch", ctypes.c_int32)]


# Diagnostics word (topk_packed_device_flags).
FLAG_STREAM_WAIT_TIMEOUT = 1
FLAG_BAD_OUTPUT_POSITION = 2
FLAG_OUT_OF_BOUNDS = 4  # checked build only; bits 8-15: the site of the first failed check
CHECK_SITES = {1: "row window leaves its buffer row", 2: "descriptor row index", 3: "window load",
               4: "window bulk copy", 5: "page-table read", 6: "page-stage read", 7: "candidate store",
               8: "region or list count", 9: "staged output position", 10: "sample load"}


def check_site(flags: int) -> int:
    """The site of the first failed bounds check recorded in a diagnostics word (0: none)."""
    return (int(flags) >> 8) & 0xFF


_libs: dict = {}
_checked = False


def library_path(checked: Optional[bool] = None) -> str:
    use = _checked if checked is None else checked
    return os.path.join(HERE, CHECKED_LIB_NAME if use else LIB_NAME)


def available(checked: bool = False) -> bool:
    return os.path.exists(library_path(checked))


@contextlib.contextmanager
def checked_build():
    """Calls made inside the block go to the bounds-checked library."""
    global _checked
    old = _checked
    _checked = True
    try:
        yield
    finally:
        _checked = old


def _load():
    lib = _libs.get(_checked)
    if lib is not None:
        return lib
    path = library_path()
    if not os.path.exists(path):
        raise TopkError(-1, f"{os.path.basename(path)} is not built (run __graft_entry__.build() or "
                            f"python -m sparse_attention_top_packed_b300.build)")
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    common = [vp, i64, vp, vp, vp, vp, i64, i32, i32, vp, i32]
    lib.topk_packed.restype = ctypes.c_int
    lib.topk_packed.argtypes = common + [vp]
    lib.topk_packed_ex.restype = ctypes.c_int
    lib.topk_packed_ex.argtypes = common + [ctypes.POINTER(LaunchConfig), vp]
    lib.topk_packed_typed.restype = ctypes.c_int
    lib.topk_packed_typed.argtypes = [vp, i32] + common[1:] + [ctypes.POINTER(LaunchConfig), vp]
    lib.topk_packed_plan.restype = ctypes.c_int
    lib.topk_packed_plan.argtypes = [i64, i32, i32, ctypes.POINTER(LaunchConfig)] + \
        [ctypes.POINTER(ctypes.c_int32)] * 4
    lib.topk_status_string.restype = ctypes.c_char_p
    lib.topk_status_string.argtypes = [ctypes.c_int]
    lib.topk_last_cuda_error.restype = ctypes.c_int
    lib.topk_last_cuda_error.argtypes = []
    lib.topk_packed_device_flags.restype = ctypes.c_int
    lib.topk_packed_device_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32, vp]
    _libs[_checked] = lib
    return lib


def _ptr(x) -> Optional[int]:
    """Device pointer of a tensor (None -> NULL; ints are taken as pointers)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch

        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int, what: str):
    if status != TOPK_OK:
        lib = _load()
        msg = lib.topk_status_string(status).decode()
        cuda = lib.topk_last_cuda_error()
        raise TopkError(status, f"{what}: {msg}" + (f" (cudaError {cuda})" if cuda else ""))


TEST_UNSATISFIED_WAIT = 1


def _config(path="auto", cluster_size: int = 0, max_ctas: int = 0,
            stream_wait_ns: int = 0, test_flags: int = 0, dependent_launch: bool = False) -> LaunchConfig:
    return LaunchConfig(PATHS[path] if isinstance(path, str) else int(path), int(cluster_size),
                        int(max_ctas), int(stream_wait_ns), int(test_flags), 1 if dependent_launch else 0)


def topk_packed(scores, row_stride: int, seq_lens, row_starts, row_to_batch, page_table,
                pt_stride: int, page_size: int, k: int, out, num_rows: int, stream=None) -> None:
    """Queues the operation on `stream` (default: torch's current stream)."""
    lib = _load()
    st = lib.topk_packed(_ptr(scores), int(row_stride), _ptr(seq_lens), _ptr(row_starts),
                         _ptr(row_to_batch), _ptr(page_table), int(pt_stride), int(page_size),
                         int(k), _ptr(out), int(num_rows), _stream_handle(stream))
    _check(st, "topk_packed")


def topk_packed_ex(scores, row_stride: int, seq_lens, row_starts, row_to_batch, page_table,
                   pt_stride: int, page_size: int, k: int, out, num_rows: int,
                   path="auto", cluster_size: int = 0, max_ctas: int = 0, stream_wait_ns: int = 0,
                   test_flags: int = 0, dependent_launch: bool = False, stream=None) -> None:
    lib = _load()
    cfg = _config(path, cluster_size, max_ctas, stream_wait_ns, test_flags, dependent_launch)
    st = lib.topk_packed_ex(_ptr(scores), int(row_stride), _ptr(seq_lens), _ptr(row_starts),
                            _ptr(row_to_batch), _ptr(page_table), int(pt_stride), int(page_size),
                            int(k), _ptr(out), int(num_rows), ctypes.byref(cfg),
                            _stream_handle(stream))
    _check(st, "topk_packed_ex")


DTYPES = {"f32": 0, "bf16": 1, "f16": 2}


def topk_packed_typed(scores, dtype: str, row_stride: int, seq_lens, row_starts, row_to_batch, page_table,
                      pt_stride: int, page_size: int, k: int, out, num_rows: int, path="auto",
                      cluster_size: int = 0, max_ctas: int = 0, dependent_launch: bool = False,
                      stream=None) -> None:
    """topk_packed_ex on a buffer of `dtype` ("f32", "bf16", "f16") elements."""
    lib = _load()
    cfg = _config(path, cluster_size, max_ctas, 0, 0, dependent_launch)
    st = lib.topk_packed_typed(_ptr(scores), DTYPES[dtype], int(row_stride), _ptr(seq_lens), _ptr(row_starts),
                               _ptr(row_to_batch), _ptr(page_table), int(pt_stride), int(page_size), int(k),
                               _ptr(out), int(num_rows), ctypes.byref(cfg), _stream_handle(stream))
    _check(st, "topk_packed_typed")


def topk_packed_plan(row_stride: int, k: int, num_rows: int, path="auto", cluster_size: int = 0,
                     max_ctas: int = 0) -> dict:
    lib = _load()
    cfg = _config(path, cluster_size, max_ctas)
    outs = [ctypes.c_int32(0) for _ in range(4)]
    st = lib.topk_packed_plan(int(row_stride), int(k), int(num_rows), ctypes.byref(cfg),
                              *[ctypes.byref(o) for o in outs])
    _check(st, "topk_packed_plan")
    names = ["path", "cluster_size", "grid_ctas", "threads_per_cta"]
    return {n: int(o.value) for n, o in zip(names, outs)}


def topk_status_string(status: int) -> str:
    return _load().topk_status_string(int(status)).decode()


def topk_packed_device_flags(reset: bool = False, stream=None) -> int:
    lib = _load()
    flags = ctypes.c_uint32(0)
    _check(lib.topk_packed_device_flags(ctypes.byref(flags), 1 if reset else 0,
                                        _stream_handle(stream)), "topk_packed_device_flags")
    return int(flags.value)


def raw_call(name: str, *args) -> int:
    """Calls a C entry point with already-marshalled arguments and returns its
    status code without raising (used to test the error paths)."""
    return int(getattr(_load(), name)(*args))


def run_workload(w, out=None, stream=None, **launch) -> "object":
    """topk_packed_ex on a Workload's tensors (all on one CUDA device)."""
    import torch

    if out is None:
        out = torch.empty((w.num_rows, w.k), dtype=torch.int32, device=w.scores.device)
    if w.scores.dtype != torch.float32:
        topk_packed_typed(w.scores, w.dtype, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch,
                          w.page_table, w.pt_stride, w.page_size, w.k, out, w.num_rows, stream=stream, **launch)
        return out
    topk_packed_ex(w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch,
                   w.page_table, w.pt_stride, w.page_size, w.k, out, w.num_rows,
                   stream=stream, **launch)
    return out
