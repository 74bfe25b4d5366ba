"""A stand-in for the kernel that writes the score buffer (the indexer in DSA
prefill), for testing and timing the dependent launch of topk_packed_ex.

The page ("[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66% 끌어올린 Top-K 커널
최적화 분석", section 2) has the top-k kernel wait on the grid that produced
its scores before reading them.  This module compiles, at run time with NVRTC,
a copy kernel that first lets its dependents start (griddepcontrol.
launch_dependents), then waits a fixed time on the global timer, then writes
the scores.  A top-k kernel launched after it with a dependent launch is
scheduled while the copy still runs, and must not read the scores before the
copy has completed.

Only the CUDA driver and NVRTC from cuda-bindings are used; the module holds
none of the top-k arithmetic.
"""
from __future__ import annotations

import ctypes

_SOURCE = rb"""
extern "C" __global__ void produce_scores(float* dst, const float* src, long long n,
                                          unsigned long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;");
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  t = t0;
  while (t - t0 < delay_ns) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}
"""

_fn = None


def _check(res, what):
    err = res[0] if isinstance(res, tuple) else res
    if int(err) != 0:
        raise RuntimeError(f"{what} failed: {err}")
    return res[1:] if isinstance(res, tuple) and len(res) > 1 else None


def _function():
    global _fn
    if _fn is not None:
        return _fn
    from cuda.bindings import driver, nvrtc

    _check(driver.cuInit(0), "cuInit")
    err, prog = nvrtc.nvrtcCreateProgram(_SOURCE, b"produce_scores.cu", 0, [], [])
    _check(err, "nvrtcCreateProgram")
    opts = [b"--gpu-architecture=sm_103a"]
    err, = nvrtc.nvrtcCompileProgram(prog, len(opts), opts)
    if int(err) != 0:
        _, n = nvrtc.nvrtcGetProgramLogSize(prog)
        log = b" " * n
        nvrtc.nvrtcGetProgramLog(prog, log)
        raise RuntimeError("NVRTC: " + log.decode(errors="replace"))
    err, size = nvrtc.nvrtcGetCUBINSize(prog)
    _check(err, "nvrtcGetCUBINSize")
    cubin = b" " * size
    _check(nvrtc.nvrtcGetCUBIN(prog, cubin), "nvrtcGetCUBIN")
    err, module = driver.cuModuleLoadData(cubin)
    _check(err, "cuModuleLoadData")
    err, fn = driver.cuModuleGetFunction(module, b"produce_scores")
    _check(err, "cuModuleGetFunction")
    _fn = fn
    return fn


def produce_scores(dst, src, delay_ns: int, stream, blocks: int = 64, threads: int = 256) -> None:
    """Queues on `stream` (a torch.cuda.Stream or raw handle) a kernel that
    copies float32 tensor `src` into `dst` (same number of elements) after
    waiting `delay_ns` nanoseconds, having first let dependents launch."""
    from cuda.bindings import driver

    if dst.numel() != src.numel():
        raise ValueError("dst and src sizes differ")
    fn = _function()
    handle = stream if isinstance(stream, int) else int(stream.cuda_stream)
    params = ((dst.data_ptr(), src.data_ptr(), int(dst.numel()), int(delay_ns)),
              (ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_ulonglong))
    _check(driver.cuLaunchKernel(fn, blocks, 1, 1, threads, 1, 1, 0, driver.CUstream(handle), params, 0),
           "cuLaunchKernel")
