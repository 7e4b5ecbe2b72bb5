"""The benchmark's reference arm (the FP64 oracle on the host cores) and its JSON line, on CPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    # value and ms_per_step describe the same timed steps: bytes per step / time per step
    sys.path.insert(0, ROOT)
    import bench
    per_step_bytes = d["value"] * 1e9 * d["ms_per_step"] / 1e3
    step_bytes = sum(bench.call_bytes(bench.CTX, n) for n in bench.N_LIVES)   # the GPU arm's step
    assert abs(per_step_bytes - step_bytes) / step_bytes < 0.01
    assert d["ms_per_step"] > 10.0   # five FP64 CPU verify calls over 196,608 positions each
    sys.path.insert(0, ROOT)
    import bench
    for k, v in bench.workload_config().items():      # the GPU arm's workload
        assert d["config"][k] == v
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
