"""Benchmark of the packed top-k + page transform.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload prefill|long|mixed|decode|tiny]

One step = one call of topk_packed over the whole workload (every row of the
batch: window load, selection, ordered emission, page transform, padding).
Default workload: the prefill chunk at ISL 70000 -- 2 requests x 70000 KV
tokens side by side (row stride 140000), the last 2048 query tokens of each
(4096 rows, windows 67953..70000 floats), k = 2048, page size 64.

Prints one JSON line.  `value` is rows/s with inputs resident in HBM (CUDA
events on the launching stream, max over ranks); `e2e` is the same metric
through the public API with pinned host buffers and the host<->device copies
in the timed region; `roofline` relates the kernel's algorithmic bytes (window
bytes read for rows with seq_len > k, plus 4*k bytes written per row) to the
measured HBM copy bandwidth; `cpu_baseline` times the CPU oracle on a bounded
sample of rows.  Under torchrun every rank runs the same workload on its own
GPU (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

WORKLOAD_TEXT = {
    "prefill": "prefill chunk ISL 70000: 4096 rows (2 requests x 2048 causal queries), "
               "row stride 140000 fp32, windows 67953..70000, k=2048, page 64",
    "long": "long context: 2048 rows, row stride 327680 fp32, windows 325633..327680, k=2048, page 64",
    "mixed": "mixed batch with ties: 16 requests (KV 1K..64K) side by side, 8192 causal rows, "
             "bf16-rounded scores, k=2048, page 64",
    "decode": "decode-like: 64 rows x 8192 fp32, k=2048, page 64",
    "tiny": "tiny: 8 rows, windows 1..300 at unaligned offsets, k=32, page 64",
    "fewlong": "few long rows: 64 rows x 327680 fp32 (fewer rows than SMs), k=2048, page 64",
    "drift": "prefill chunk ISL 70000 with drifting scores: row q of a request holds N(0,1)*s_q + m_q, "
             "m_q = 0.5 sin(2 pi q/300) + 0.05 N(0,1), s_q = 1 + 0.25 sin(2 pi q/450), k=2048, page 64",
}
L2_BYTES = 126 * 1024 * 1024


def log(msg: str) -> None:
    print(msg, file=sys.stderr, flush=True)


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured", "sm_max_mhz": d.get("sm_max_mhz")}
    return {"hbm_gbs": 6400.0, "source": "fallback", "sm_max_mhz": 2032.0}


def _code_only(text: str) -> str:
    """C++ source without its comments and blank lines (no string literal in
    the kernel sources holds a comment marker)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash() -> str:
    """First 16 hex digits of the sha256 of the kernel sources' code (file
    names and contents, comments and blank lines left out): it changes when the
    kernels do, not when a comment does."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_top_packed_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(workload)
    if not entry or entry.get("source_hash") != kernel_source_hash():
        return None
    return entry.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sm, mem, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if self.t0 is None or not (self.t0 - 0.15 <= t <= self.t1 + 0.15):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                if len(parts) > 9:
                    mem.append(float(parts[9]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "mem_mhz": statistics.median(mem) if mem else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def make_workload(name: str, device, rows: int = 0, dtype: str = "f32"):
    from sparse_attention_top_packed_b300 import workloads

    w = workloads.named(name, device=device)
    w = w.head(rows) if rows else w
    return w if dtype == "f32" else workloads.with_dtype(w, dtype)


def l2_flush_buffer(device):
    return torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)


def make_launch(path: str, dtype: str = "f32"):
    """The timed call: topk_packed (the automatic choice), topk_packed_ex with
    an explicit kernel family, or topk_packed_typed for a 16-bit buffer."""
    from sparse_attention_top_packed_b300 import binding

    if dtype != "f32":
        return lambda args, stream: binding.topk_packed_typed(args[0], dtype, *args[1:], path=path, stream=stream)
    if path == "auto":
        return lambda args, stream: binding.topk_packed(*args, stream=stream)
    return lambda args, stream: binding.topk_packed_ex(*args, path=path, stream=stream)


def prepare_timing(w, steps: int, warmup: int, flush: bool, device, launch):
    """Arguments of the timed call, after `warmup` untimed calls, and the events."""

    out = torch.empty((w.num_rows, w.k), dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    scratch = l2_flush_buffer(device) if flush else None
    args = (w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch, w.page_table,
            w.pt_stride, w.page_size, w.k, out, w.num_rows)
    for _ in range(warmup):
        if flush:
            scratch.fill_(1.0)
        launch(args, stream)
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    return args, stream, scratch, starts, ends


def device_copy_gbs(device, nbytes: int = 1 << 29, reps: int = 5) -> float:
    """This GPU's plain copy rate right now (read + write bytes of a 512 MB
    torch copy, best of `reps`, CUDA events): context for the roofline,
    whose peak is the pool's measured figure."""
    a = torch.empty(nbytes // 4, dtype=torch.float32, device=device).fill_(1.0)
    b = torch.empty_like(a)
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize(device)
        best = min(best, e0.elapsed_time(e1))
    del a, b
    return 2 * nbytes / (best / 1e3) / 1e9


def run_ours(a, rank: int, world: int, device) -> dict:
    from sparse_attention_top_packed_b300 import binding

    torch.cuda.set_device(device)
    w = make_workload(a.workload, device, a.rows, a.dtype)
    torch.cuda.synchronize(device)
    alg_bytes = w.algorithmic_bytes()
    big = w.window_bytes() > 4 * L2_BYTES
    flush = not big
    launch = make_launch(a.path, a.dtype)
    args, stream, scratch, starts, ends = prepare_timing(w, a.steps, a.warmup, flush, device, launch)
    if a.graph:
        # the launch captured once in a CUDA graph; the timed steps replay it
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            launch(args, torch.cuda.current_stream(device))
        for _ in range(a.warmup):
            graph.replay()
        torch.cuda.synchronize(device)
        launch = lambda args_, stream_: graph.replay()  # noqa: E731

    copy_gbs = device_copy_gbs(device)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(1.0)  # nvidia-smi needs a moment before its first sample
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark_begin()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(a.steps):
        if flush:
            scratch.fill_(1.0)
        starts[i].record(stream)
        launch(args, stream)
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    if sampler:
        sampler.mark_end()
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_ms = sum(launch_ms) / len(launch_ms)
    step_ms = kernel_ms if flush else t_begin.elapsed_time(t_end) / a.steps
    clocks = sampler.stop() if sampler else None

    # max over ranks
    if world > 1:
        t = torch.tensor([step_ms, kernel_ms], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        step_ms, kernel_ms = float(t[0]), float(t[1])

    # the diagnostics word after the timed launches: a bounded wait that gave
    # up would show here (the run is then rejected)
    flags = binding.topk_packed_device_flags(reset=True)
    out = args[9]
    e2e = run_e2e(a, w, device) if rank == 0 else None
    result = {
        "step_ms": step_ms, "kernel_ms": kernel_ms, "alg_bytes": alg_bytes, "flush": flush,
        "clocks": clocks, "e2e": e2e, "workload": w, "out": out, "device_flags": flags, "copy_gbs": copy_gbs,
    }
    return result


def run_e2e(a, w, device) -> dict:
    """Same metric through the public API with pinned host buffers: each step
    copies the step's inputs host->device, runs topk_packed, copies the result
    back.  Timed with CUDA events on the stream doing all three."""
    from sparse_attention_top_packed_b300 import binding

    steps = max(1, min(a.steps, a.e2e_steps))
    host = {}
    for name in ("scores", "seq_lens", "row_starts", "row_to_batch", "page_table"):
        t = getattr(w, name)
        if t is not None:
            host[name] = t.cpu().pin_memory()
    dev = {n: torch.empty_like(t, device=device) for n, t in host.items()}
    out_dev = torch.empty((w.num_rows, w.k), dtype=torch.int32, device=device)
    out_host = torch.empty((w.num_rows, w.k), dtype=torch.int32).pin_memory()
    stream = torch.cuda.current_stream(device)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * 4

    launch = make_launch(a.path, a.dtype)

    def step():
        for n in host:
            dev[n].copy_(host[n], non_blocking=True)
        launch((dev["scores"], w.row_stride, dev["seq_lens"], dev["row_starts"], dev.get("row_to_batch"),
                dev["page_table"], w.pt_stride, w.page_size, w.k, out_dev, w.num_rows), stream)
        out_host.copy_(out_dev, non_blocking=True)

    step()
    torch.cuda.synchronize(device)
    b = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    b.record(stream)
    for _ in range(steps):
        step()
    e.record(stream)
    torch.cuda.synchronize(device)
    ms = b.elapsed_time(e) / steps
    return {"value": w.num_rows / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms, "steps": steps}


def oracle_sample(w, n: int, seed: int):
    """Host copies of the windows of a sample of n rows (first, last and
    evenly spread), and the arguments the CPU oracle takes for them."""
    from sparse_attention_top_packed_b300.workloads import gather_windows, sample_rows

    rows = sample_rows(w.num_rows, n, seed=seed)
    win, L = gather_windows(w, rows)
    b = (rows.numpy() if w.row_to_batch is None
         else w.row_to_batch[rows.to(w.row_to_batch.device)].cpu().numpy()).astype(np.int32)
    table = w.page_table.reshape(-1).cpu().numpy()
    return rows, (win.reshape(-1), win.shape[1], L, np.zeros(len(L), np.int32), b, table,
                  w.pt_stride, w.page_size, w.k)


def time_oracle(args, cores: int):
    """One call of the CPU oracle as it stands (all rows of the sample, `cores`
    threads): seconds and its [rows, k] result."""
    from oracle import topk_packed_reference

    t0 = time.perf_counter()
    res = topk_packed_reference(*args, nthreads=cores)
    return time.perf_counter() - t0, res


def cpu_baseline(w, out, target_s: float = 12.0) -> dict:
    """The CPU oracle, as it stands, on a bounded sample of the workload's rows
    (windows copied to the host first, outside the timing), all host cores,
    in one call.  A small probe sizes the sample to about `target_s` seconds
    of oracle work, or the whole workload when that takes less.  The oracle's
    result for those rows is also compared with the timed launch's output
    (`spot_check`)."""
    from oracle import default_threads

    cores = default_threads()
    rows, args = oracle_sample(w, min(w.num_rows, max(2 * cores, 16)), seed=1)
    dt, res = time_oracle(args, cores)
    n = int(rows.numel())
    if n < w.num_rows:
        want = int(n * target_s / max(dt, 1e-4))
        n2 = min(w.num_rows, max(n, want))
        if n2 > n:
            del args, res
            rows, args = oracle_sample(w, n2, seed=1)
            dt, res = time_oracle(args, cores)
            n = int(rows.numel())
    got = out[rows.to(out.device)].cpu().numpy()
    bad = int((got != res).any(axis=1).sum())
    return {"value": n / dt, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.num_rows} rows (first, last and evenly spread) in one call, "
                      f"{dt:.2f} s on {cores} threads; windows copied to the host beforehand",
            "spot_check": {"rows": n, "mismatched_rows": bad,
                           "what": "the timed launch's output rows against the oracle's, int32 equality"}}


def run_pdl_gap(a, device) -> None:
    """Times pairs of (producer kernel, topk_packed_ex) on one stream, with and
    without the dependent launch, and prints one JSON line.  The producer is a
    stand-in for the kernel writing the scores (a copy of them, no added
    delay) that lets its dependents start at once."""
    from sparse_attention_top_packed_b300 import binding
    from sparse_attention_top_packed_b300.producer import produce_scores

    torch.cuda.set_device(device)
    w = make_workload(a.workload, device, a.rows)
    src = w.scores.clone()
    out = torch.empty((w.num_rows, w.k), dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device)
    args = (w.scores, w.row_stride, w.seq_lens, w.row_starts, w.row_to_batch, w.page_table,
            w.pt_stride, w.page_size, w.k, out, w.num_rows)
    res = {}
    for dep in (False, True, False, True):
        def pair():
            produce_scores(w.scores, src, 0, stream)
            binding.topk_packed_ex(*args, path=a.path, dependent_launch=dep, stream=stream)
        for _ in range(a.warmup):
            pair()
        stream.synchronize()
        b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b.record(stream)
        for _ in range(a.steps):
            pair()
        e.record(stream)
        stream.synchronize()
        res.setdefault(dep, []).append(b.elapsed_time(e) * 1e3 / a.steps)
    plain, dep = min(res[False]), min(res[True])
    print(json.dumps({"pdl_gap": {"workload": WORKLOAD_TEXT[a.workload], "pairs": a.steps,
                                  "us_per_pair_plain": plain, "us_per_pair_dependent": dep,
                                  "saving_us": plain - dep,
                                  "what": "producer kernel (score copy) then topk_packed_ex on one stream, "
                                          "CUDA events over the pairs, best of two runs"}}), flush=True)


def run_reference(a, rank: int, world: int) -> None:
    """The reference arm: the CPU oracle, timed as it stands on the host cores,
    on the same workload and metric.  Every step is one call of the oracle on
    the same bounded sample of rows (about 512 MB of windows), as in the
    cpu_baseline leg, so the two figures measure the same thing."""
    if rank != 0:
        return
    from oracle import default_threads

    device = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    w = make_workload(a.workload, device, a.rows, a.dtype)
    cores = default_threads()
    avg_row_bytes = max(w.window_bytes_all() / max(w.num_rows, 1), 4.0)
    rows_per_step = int(min(w.num_rows, max(16 * cores, (512 << 20) // avg_row_bytes)))
    rows, args = oracle_sample(w, rows_per_step, seed=1)
    rows_per_step = int(rows.numel())
    steps = []
    for s in range(a.warmup + a.steps):
        dt, _ = time_oracle(args, cores)
        if s >= a.warmup:
            steps.append(dt)
    sec = sum(steps) / len(steps)
    value = rows_per_step / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config_block(a, w, None),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"the same {rows_per_step} of {w.num_rows} rows every step, one call each"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


KERNEL_NAMES = {1: "topk_multipass_kernel", 2: "topk_stream_kernel", 3: "topk_pipe_kernel", 4: "topk_split_kernel",
                5: "topk_decode_kernel"}
METRIC = "packed top-k rows/s and achieved HBM GB/s (% of B300 peak), 1 GPU"


def config_block(a, w, plan) -> dict:
    d = {"workload": WORKLOAD_TEXT[a.workload] + ("" if w.dtype == "f32" else f", scores held as {w.dtype}"),
         "rows": w.num_rows, "row_stride": w.row_stride,
         "k": w.k, "page_size": w.page_size,
         "window_bytes_per_step": w.window_bytes(), "output_bytes_per_step": w.output_bytes(),
         "l2": ("inputs larger than L2: each step reads %.2f GB, no flush" % (w.window_bytes() / 1e9))
         if w.window_bytes() > 4 * L2_BYTES else "L2 flushed (252 MB write) before every timed launch",
         "parallelism": f"dp{a.gpus} (independent replicas of the batch)"}
    if plan is not None:
        d["launch"] = plan
    if getattr(a, "graph", False):
        d["timing"] = "each step replays a CUDA graph holding the launch"
    return d


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--rows", type=int, default=0,
                    help="keep only the first N rows of the workload (small profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "pipe", "split", "stream", "multipass", "decode"],
                    help="kernel family (auto: the choice topk_packed makes)")
    ap.add_argument("--dtype", default="f32", choices=["f32", "bf16", "f16"],
                    help="element type of the score buffer (16-bit: the values rounded to it)")
    ap.add_argument("--graph", action="store_true",
                    help="capture the launch in a CUDA graph and time graph replays")
    ap.add_argument("--pdl-gap", action="store_true",
                    help="time producer + top-k pairs with and without the dependent launch instead")
    a = ap.parse_args()
    if a.warmup < 3:
        a.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if a.impl == "reference":
        run_reference(a, rank, world)
        return
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if a.pdl_gap:
        if rank == 0:
            run_pdl_gap(a, device)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)

    from sparse_attention_top_packed_b300 import binding

    r = run_ours(a, rank, world, device)
    w = r["workload"]
    mismatched = 0
    if rank == 0:
        peaks = measured_peaks()
        plan = binding.topk_packed_plan(w.row_stride, w.k, w.num_rows, path=a.path)
        achieved = r["alg_bytes"] / (r["kernel_ms"] / 1e3) / 1e9
        value = world * w.num_rows / (r["step_ms"] / 1e3)
        traffic = profiled_traffic(a.workload)
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": r["step_ms"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded N(0,1) scores, distinct random pages)",
            "config": config_block(a, w, plan),
            "achieved_hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)"
                         if peaks["source"] == "measured" else "fallback 6.4 TB/s",
                         "algorithmic_bytes_per_launch": r["alg_bytes"],
                         "kernel": KERNEL_NAMES.get(plan["path"], "?"),
                         "device_copy_gbs": r["copy_gbs"],
                         "device_copy_note": "this GPU's 512 MB torch copy rate (read+write bytes, best of 5) "
                                             "just before the timed region; the peak above is the pool's"},
            "gpu_launches": a.steps,
            "clocks": r["clocks"],
            "e2e": r["e2e"],
            "device_flags": r["device_flags"],
        }
        if world == 1 and not a.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, r["out"])
            mismatched = line["cpu_baseline"]["spot_check"]["mismatched_rows"]
        print(json.dumps(line), flush=True)
    failed = r["device_flags"] != 0 or bool(mismatched)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if failed:
        log("bench: the timed output failed its check (diagnostics word or oracle spot check); see the JSON line")
        sys.exit(1)


if __name__ == "__main__":
    main()
