"""The small parity cases under the debug build (the stand-in for a memory checker).

The debug build (WCOMP_DEBUG=1) checks indexes before the kernels' memory
accesses: escape positions against the tensor and its rows, decode and GEMV
outputs and x reads against their buffers, encoder stash and escape-stream
indexes.  A failed check skips the access and is reported by
wcomp_device_check as WCOMP_EBOUNDS.  Here the encoder, decode, fused and
plain GEMV run through that build on edge cases (every BF16 pattern, ragged
sizes, escapes on row and tile boundaries, partial k-blocks and units,
batches) in a child process, each checked against the oracle, and no check
may fire.

The same build also makes the GEMV kernels' bounded waits run out without a
fault: with the skip hook on, every warp leaves its first tensor copy
unissued and waits for it (nothing will complete that wait), gives up after
about a second, and the launch must report WCOMP_ETIMEOUT; with the hook off
the next launch on the same context must be correct and report nothing.
"""
import os
import subprocess
import sys

import pytest

pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from decode_gemv_sign_gb300 import synth, wcomp as W
from oracle import wcomp_oracle as O
W.LIB_PATH = sys.argv[2]
W.lib()

def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()

cases = [
    np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256),
    np.random.default_rng(3).integers(0, 65536, size=(3, 11)).astype(np.uint16),
    synth.gen_weights_np(synth.WeightSpec("r", 7, 301, "t4", 0.02, 0.01, "normal", 1.0, seed=11)),
    synth.gen_weights_np(synth.WeightSpec("r", 3, 40000, "t4", 0.02, 0.01, "normal", 1.0, seed=12)),
    synth.gen_weights_np(synth.WeightSpec("g", 37, 2048, "t4", 0.02, 0.02, "normal", 1.0, seed=13)),
    synth.gen_weights_np(synth.WeightSpec("g", 130, 1056, "t4", 0.02, 0.02, "normal", 1.0, seed=14)),
    synth.gen_weights_np(synth.WeightSpec("g", 64, 4096, "t4", 0.02, 0.05, "normal", 1.0, seed=15)),
]
checked = 0
for w in cases:
    N, K = w.shape
    for scheme in O.SCHEMES:
        ref = O.encode(w, scheme)
        c = W.encode(dev(w), scheme)
        assert W.serialize(c) == O.serialize(ref)
        assert np.array_equal(W.decode(c).cpu().numpy().view(np.uint16).reshape(w.shape), w)
        for B in (1, 2, 4, 8, 9, 16):
            x = synth.gen_x_np(B, K, 50 + B)
            y = W.gemv(c, dev(x)).cpu().numpy().astype(np.float64)
            yn = torch.empty((B, N), dtype=torch.float32, device="cuda")
            W.gemv_noalloc(c, dev(x), yn)
            yr = O.gemv(w, x)
            if np.isfinite(yr).all():  # the all-patterns case holds Inf and NaN weights
                assert np.abs(y - yr).max() <= 1e-4 * max(np.abs(yr).max(), 1e-30)
                assert np.abs(yn.cpu().numpy().astype(np.float64) - yr).max() <= 1e-4 * max(np.abs(yr).max(), 1e-30)
                checked += 1
        c.free()
    for B in (1, 8, 16):
        x = synth.gen_x_np(B, K, 90 + B)
        y = W.gemv_bf16(dev(w), dev(x)).cpu().numpy().astype(np.float64)
        yr = O.gemv(w, x)
        if np.isfinite(yr).all():
            assert np.abs(y - yr).max() <= 1e-4 * max(np.abs(yr).max(), 1e-30)
ws = [cases[4], cases[5], cases[6]]
cs = W.encode_batched([dev(w) for w in ws for _ in (0, 1)], [0, 1] * len(ws))
outs = W.decode_batched(cs)
for i, o in enumerate(outs):
    assert np.array_equal(o.cpu().numpy().view(np.uint16).reshape(ws[i // 2].shape), ws[i // 2])
xs = [dev(synth.gen_x_np(4, w.shape[1], 70 + i)) for i, w in enumerate(ws) for _ in (0, 1)]
W.gemv_batched(cs, xs)
torch.cuda.synchronize()
st = W.lib().wcomp_device_check(None)
print("device_check", st, "checked", checked)
sys.exit(0 if st == 0 else 3)
"""


def test_parity_cases_under_the_debug_build():
    from decode_gemv_sign_gb300 import build

    lib = build.build(debug=True)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, lib], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "device_check 0" in r.stdout


TIMEOUT_CHILD = r"""
import sys, time
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from decode_gemv_sign_gb300 import synth, wcomp as W
from oracle import wcomp_oracle as O
W.LIB_PATH = sys.argv[2]
L = W.lib()

def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()

w = synth.gen_weights_np(synth.WeightSpec("g", 96, 2048, "t4", 0.02, 0.02, "normal", 1.0, seed=21))
N, K = w.shape
assert L.wcomp_device_check(None) == W.OK
for scheme in O.SCHEMES:
    c = W.encode(dev(w), scheme)
    for B in (1, 4):
        x = synth.gen_x_np(B, K, 30 + B)
        yr = O.gemv(w, x)
        for plain in (False, True):
            assert L.wcomp_debug_skip_first_copy(1) == W.OK
            t0 = time.time()
            y = W.gemv_bf16(dev(w), dev(x)) if plain else W.gemv(c, dev(x))
            torch.cuda.synchronize()
            dt = time.time() - t0
            st = L.wcomp_device_check(None)
            assert st == W.ETIMEOUT, (scheme, B, plain, st)
            assert 0.5 < dt < 30, dt
            assert L.wcomp_debug_skip_first_copy(0) == W.OK
            y = W.gemv_bf16(dev(w), dev(x)) if plain else W.gemv(c, dev(x))
            y = y.cpu().numpy().astype(np.float64)
            assert L.wcomp_device_check(None) == W.OK
            assert np.abs(y - yr).max() <= 1e-4 * np.abs(yr).max()
            print("timed out and recovered", scheme, B, plain, round(dt, 2))
    c.free()
print("ok")
"""


def test_bounded_waits_run_out_and_report_etimeout():
    from decode_gemv_sign_gb300 import build

    lib = build.build(debug=True)
    r = subprocess.run([sys.executable, "-c", TIMEOUT_CHILD, ROOT, lib], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("timed out and recovered") == 8 and "ok" in r.stdout
