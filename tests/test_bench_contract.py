"""bench.py's reference arm (the fp64 oracle on the host cores) runs here on
the CPU: its one JSON line must carry the keys and relations of the benchmark
contract that the GPU arm's line carries too (CPU)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])

    sys.path.insert(0, ROOT)
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "us/token" and d["higher_is_better"] is False
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 1, 3)
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["dtype"] == "f64"
    assert d["config"]["workload"].startswith("llama2-7b-reglu-decode")
    assert (d["config"]["d_model"], d["config"]["d_ff"], d["config"]["batch"]) == (4096, 11008, 1)
    # value = the step's time over the tokens it decoded
    per_step = d["config"]["tokens_per_step"]
    assert per_step >= 1 and d["value"] > 0
    assert abs(d["value"] - d["ms_per_step"] * 1e3 / per_step) <= 0.01 * d["value"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and isinstance(cb["sample"], str) and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
