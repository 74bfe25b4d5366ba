"""bench.py's reference arm on the CPU: one JSON line with the keys the
benchmark contract names, the oracle as the timed program, and the end-to-end
object describing a host-only run."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    proc = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                           "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [l for l in proc.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, proc.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    # at least 3 warm-up steps, whatever was asked
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["unit"] == "rows/s" and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_profiles_describe_the_current_kernels():
    """profiles/dram_traffic.json was captured on the kernel code in the tree
    (its hash leaves comments out), so the bench reports the measured traffic."""
    sys.path.insert(0, ROOT)
    import bench

    assert bench._code_only("a; // note\n/* block\n comment */b;\n\n  c;  // x") == "a;\nb;\n  c;"
    for workload in ("prefill", "long", "fewlong", "decode"):
        assert bench.profiled_traffic(workload), workload
