"""wcomp_gemv_noalloc: the GEMV entry point that allocates nothing.

It serves callers that cannot let the library allocate device memory (a fixed
memory budget, or no implicit synchronisation from cudaMalloc / cudaFree); its
work counters live in a small static device array instead of a buffer the
library allocates.  Checked through the C ABI against wcomp_gemv on the same
container and input, and against the CPU oracle's float64 GEMV, on two calls
in a row (the array keeps the previous call's contents, so the second call
shows that the counters are cleared).

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test first; it also passes on its own in a fresh
process.
"""
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("scheme", [0, 1])
@pytest.mark.parametrize("B", [1, 4, 16])
@pytest.mark.parametrize("shape", [(300, 2048), (37, 1000), (41, 2080)])
def test_noalloc_matches_gemv_twice(W, scheme, B, shape):
    N, K = shape
    w = synth.gen_weights_np(synth.WeightSpec("na", N, K, "t4", 0.02, 0.01, "normal", 1.0, seed=7000 + B + N))
    x = synth.gen_x_np(B, K, 7100 + B)
    c = W.encode(dev(w), scheme)
    xd = dev(x)
    y_lib = W.gemv(c, xd).cpu().numpy().astype(np.float64)
    y_ora = O.gemv(w, x)
    scale = np.abs(y_ora).max()
    assert np.abs(y_lib - y_ora).max() <= GEMV_TOL * scale
    for _ in range(2):
        y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
        W.gemv_noalloc(c, xd, y)
        got = y.cpu().numpy().astype(np.float64)
        assert np.abs(got - y_lib).max() <= GEMV_TOL * scale
        assert np.abs(got - y_ora).max() <= GEMV_TOL * scale
    W.device_check()
    c.free()


def test_noalloc_rejects_bad_arguments(W):
    c = W.encode(dev(np.zeros((4, 64), np.uint16)), 0)
    y = torch.zeros((17, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(W.WcompError):
        W.gemv_noalloc(c, torch.zeros((17, 64), dtype=torch.int16, device="cuda"), y)
    c.free()
