"""The benchmark's reference arm on the host: one JSON line in the same terms as ours.

The reference arm is the CPU oracle timed on the host cores; it must report
the same metric, unit, direction and workload config as the GPU arm, plus a
cpu_baseline describing the run and an e2e object with no host/device bytes.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from decode_gemv_sign_gb300 import synth  # noqa: E402


def test_reference_arm_line_matches_our_terms():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"] == bench.workload_config(synth.workload_dense_layers(), 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["vs_baseline"] is None


def test_workload_config_counts_the_dense_layer_set():
    specs = synth.workload_dense_layers()
    cfg = bench.workload_config(specs, 4)
    assert cfg["tensors"] == 7
    assert cfg["elements"] == 4 * 4096 * 4096 + 3 * 4096 * 11008 == 202375168
    assert cfg["batches"] == [1, 4] and cfg["parallelism"] == "replicas x4"
