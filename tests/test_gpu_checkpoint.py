"""Checkpoint-shaped workload (the 120 GiB, 1,923-tensor recipe) on the GPU.

1. Streamed validation in HBM-sized batches: every tensor round-trips bit for
   bit in both schemes (the pages' exactness criterion), the accounting lands
   near the pages' figures, and a rerun with the result log resumes without
   redoing work.
2. Container bytes equal the CPU oracle's for one tensor of each small shape.
3. The 16384x53248 GEMV at batch 1..16: sampled rows against the oracle's
   float64 GEMV on the exact weights (the container is lossless, checked by
   its own round trip).
"""
import json
import os

import numpy as np
import pytest

from decode_gemv_sign_gb300 import synth
from oracle import wcomp_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMV_TOL = 1e-4


@pytest.fixture(scope="module")
def W():
    from decode_gemv_sign_gb300 import build, wcomp

    build.build()
    wcomp.lib()
    return wcomp


def host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def test_checkpoint_streamed_full(W, tmp_path):
    from decode_gemv_sign_gb300 import validate

    specs = synth.workload_checkpoint()
    assert len(specs) == 1923
    assert abs(synth.total_elements(specs) * 2 / 2**30 - 120.0) < 0.01
    log = str(tmp_path / "ckpt.jsonl")
    res = validate.validate(specs, (0, 1), batch_bytes=16 << 30, log_path=log)
    for name, r in res["schemes"].items():
        assert r["tensors"] == 1923
        assert r["not_exact"] == [], name
    bs, k15 = res["schemes"]["bytesplit"], res["schemes"]["k15"]
    # the pages' accounting on their checkpoint: 12.005 and 11.173 bits/weight;
    # this synthetic set has heavier tails in half its tensors, so only the range is fixed
    assert 12.0 < bs["entropy_bpw"] < 12.05
    assert 11.1 < k15["entropy_bpw"] < 11.35
    assert bs["physical_bpw"] < 12.1
    # the compact form's physical size tracks the accounting (no positions, 9-bit K15 symbols)
    assert bs["physical_compact_bpw"] - bs["entropy_bpw"] < 0.02
    assert k15["physical_compact_bpw"] - k15["entropy_bpw"] < 0.02
    # resume: everything is in the log, nothing is redone
    lines = open(log).read().splitlines()
    assert len(lines) == 2 * 1923
    again = validate.validate(specs, (0, 1), batch_bytes=16 << 30, log_path=log)
    assert len(open(log).read().splitlines()) == 2 * 1923
    assert again["schemes"] == res["schemes"]


def test_checkpoint_small_shapes_match_oracle(W):
    specs = synth.workload_checkpoint(layers=1)
    dev = torch.device("cuda")
    chosen = {}
    for s in specs:
        if (s.N, s.K) in ((2048, 6144), (6144, 6144), (1, 6144)) and (s.N, s.K) not in chosen:
            chosen[(s.N, s.K)] = s
    assert len(chosen) == 3
    for s in chosen.values():
        w = synth.gen_weights_torch(s, dev)
        w_np = host(w).reshape(s.N, s.K)
        for scheme in O.SCHEMES:
            c = W.encode(w, scheme)
            ref = O.encode(w_np, scheme)
            assert W.serialize(c) == O.serialize(ref)
            assert W.serialize(c, compact=True) == O.serialize_compact(ref)
            c.free()


def test_checkpoint_gemv_16384x53248(W):
    dev = torch.device("cuda")
    spec = synth.checkpoint_gemv_spec()
    w = synth.gen_weights_torch(spec, dev)
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(spec.N, size=24, replace=False))
    w_rows = host(w[torch.from_numpy(rows).to(dev)]).reshape(len(rows), spec.K)
    for scheme in O.SCHEMES:
        c = W.encode(w, scheme)
        out = W.decode(c)
        assert torch.equal(out.view(-1), w.view(-1))
        del out
        for B in (1, 2, 4, 8, 16):
            x = synth.gen_x_np(B, spec.K, 6000 + B)
            y = W.gemv(c, torch.from_numpy(x.view(np.int16)).to(dev)).cpu().numpy()[:, rows].astype(np.float64)
            y_ref = O.gemv(w_rows, x)
            assert np.abs(y - y_ref).max() <= GEMV_TOL * np.abs(y_ref).max()
        c.free()
    W.device_check()


def test_streamed_from_pinned_host_with_hashes_and_corruption(W, tmp_path):
    """One layer of the checkpoint-shaped set streamed from pinned host memory in
    256 MiB batches (each batch copied while the previous one is processed):
    every tensor round-trips, its decoded bytes hash like its source in both
    schemes, every injected single-byte corruption is refused by the
    deserializer, and a log cut short mid-record resumes with only that tensor
    redone."""
    from decode_gemv_sign_gb300 import validate

    specs = [s for s in synth.workload_checkpoint(layers=1) if s.N != 151552]
    assert len(specs) == 17
    log = str(tmp_path / "host.jsonl")
    res = validate.validate(specs, (0, 1), batch_bytes=256 << 20, log_path=log, source="host", hashes=True,
                            corrupt_every=3)
    assert res["source"] == "host"
    for name, r in res["schemes"].items():
        assert r["tensors"] == 17
        assert r["not_exact"] == [], name
        assert r["hashed"] == 17 and r["hash_mismatch"] == [], name
        assert r["corruption_checks"] == 2 * len(range(0, 17, 3)) and r["corruption_missed"] == 0, name
    recs = [json.loads(line) for line in open(log)]
    assert all(r["source_hash"] == r["decoded_hash"] for r in recs)
    # the same tensor hashes the same in both schemes (one source)
    by = {}
    for r in recs:
        by.setdefault(r["name"], set()).add(r["source_hash"])
    assert all(len(v) == 1 for v in by.values())
    # an interruption in the middle of the last record: that record is dropped and redone
    data = open(log).read()
    cut = data.rstrip("\n").rfind("\n") + 1
    open(log, "w").write(data[:cut + 20])
    again = validate.validate(specs, (0, 1), batch_bytes=256 << 20, log_path=log, source="host", hashes=True)
    assert len(open(log).read().splitlines()) == 2 * 17
    assert again["schemes"]["bytesplit"]["not_exact"] == [] and again["schemes"]["k15"]["not_exact"] == []
