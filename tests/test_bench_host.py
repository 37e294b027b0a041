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
import pytest  # noqa: E402
from decode_gemv_sign_gb300 import synth  # noqa: E402
from oracle import wcomp_oracle as O  # noqa: E402


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
    assert d["config"] == bench.workload_config(synth.checkpoint_batch(0, bench.BATCH_BYTES),
                                                synth.checkpoint_gemv_spec(), 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["vs_baseline"] is None


def test_workload_config_counts_the_checkpoint_batch():
    """One step covers the first HBM-sized (16 GiB) batch of the checkpoint-shaped
    set: both embeddings and the first layers, and the 16384x53248 GEMV."""
    specs = synth.checkpoint_batch(0, bench.BATCH_BYTES)
    cfg = bench.workload_config(specs, synth.checkpoint_gemv_spec(), 4)
    assert cfg["tensors"] == len(specs) == 208
    assert 2 * cfg["elements"] <= bench.BATCH_BYTES < 2 * cfg["elements"] + 2 * 16384 * 6144
    assert [(s.N, s.K) for s in specs[:2]] == [(151552, 6144)] * 2
    assert cfg["gemv"] == [16384, 53248]
    assert cfg["batches"] == [1, 4, 8, 16] and cfg["parallelism"] == "replicas x4"
    # the batches of the whole set cover all 1,923 tensors in order
    groups = synth.batches(synth.workload_checkpoint(), bench.BATCH_BYTES)
    assert groups[0] == specs and sum(len(g) for g in groups) == 1923


def _info(c) -> dict:
    """The fields of wcomp_info that the byte counts use, for an oracle container
    (section sizes padded to 32 bytes, as the library reports them)."""
    pad = lambda x: (x + 31) // 32 * 32  # noqa: E731
    sec = dict(O.section_sizes(c.scheme, c.N, c.K, c.E))
    raw = pad(sec["raw"]) if c.scheme == O.BYTESPLIT else sum(pad(sec[k]) for k in ("plane_a", "plane_b", "plane_c"))
    return {"scheme": c.scheme, "N": c.N, "K": c.K, "n": c.n, "n_tiles": c.n_tiles, "n_escapes": c.E,
            "bytes_codes": pad(sec["codes"]), "bytes_raw": raw, "serialized_bytes": len(O.serialize(c))}


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_algorithmic_bytes_per_weight(scheme):
    """The roofline numerator against the format's per-weight sizes: a 4-bit code,
    8 raw bits (byte-split) or 7 (K15), 16 bits written by decode, and per escape
    a 4-byte position plus its 2-byte value (the device keeps whole escape
    words for both schemes)."""
    spec = synth.WeightSpec("d", 1024, 2048, "normal", 0.02, 0.001, "normal", 0.5, seed=3)
    c = O.encode(synth.gen_weights_np(spec), scheme)
    inf = _info(c)
    n, E = c.n, c.E
    assert E > 0
    raw = 1.0 if scheme == O.BYTESPLIT else 7 / 8
    esc = 6
    tiles = 4 * (c.n_tiles + 1) / n
    rows = 4 * (c.N + 1) / n
    assert bench.decode_bytes(inf) / n == pytest.approx(0.5 + raw + 2 + esc * E / n + tiles, abs=1e-12)
    for B in (1, 4, 16):
        io = (2 * B * c.K + 4 * B * c.N) / n
        assert bench.gemv_bytes(inf, B) / n == pytest.approx(0.5 + raw + esc * E / n + rows + io, abs=1e-12)
        assert bench.plain_bytes(c.N, c.K, B) / n == pytest.approx(2 + io, abs=1e-12)
    # encode reads the source once and writes the container once (header excluded)
    assert bench.encode_bytes(inf) == 2 * n + len(O.serialize(c)) - 96
