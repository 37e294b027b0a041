"""The dense 12-bit ablation workload on the GPU: escape-free weights.

The pages' GPU prototype read dense 12-bit codes with escapes handled apart
("Prueba de GLM-5.2 reduce la memoria BF16 en casi un 25%", section "Qué
queda por demostrar").  On weights whose every high byte is in the table the
byte-split container is exactly that: 4 code bits and 8 raw bits per weight,
no escape stream.  The library's container must then equal the oracle's, and
the fused GEMV (which then corrects nothing) must match the float64 oracle;
the benchmark times this case beside the escaped workload.
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


def test_dense12_container_and_gemv_small(W):
    w = synth.gen_weights_np(synth.dense12_spec(96, 4096, seed=6001))
    ref = O.encode(w, O.BYTESPLIT)
    assert ref.E == 0
    c = W.encode(dev(w), O.BYTESPLIT)
    assert c.info()["n_escapes"] == 0
    assert W.serialize(c) == O.serialize(ref)
    assert np.array_equal(W.decode(c).cpu().numpy().view(np.uint16).reshape(w.shape), w)
    for B in (1, 4, 16):
        x = synth.gen_x_np(B, 4096, 6100 + B)
        y = W.gemv(c, dev(x)).cpu().numpy().astype(np.float64)
        y_ref = O.gemv(w, x)
        assert np.abs(y - y_ref).max() <= GEMV_TOL * np.abs(y_ref).max()
    c.free()


def test_dense12_full_size_sampled_rows(W):
    """The benchmark's escape-free 16384x53248 weight: no escapes, exact round
    trip, GEMV rows against the oracle."""
    spec = synth.dense12_spec()
    w = synth.gen_weights_torch(spec, torch.device("cuda"))
    c = W.encode(w, O.BYTESPLIT)
    assert c.info()["n_escapes"] == 0
    assert abs(c.info()["entropy_bpw"] - 12.0) < 1e-4
    out = W.decode(c)
    assert torch.equal(out, w)
    del out
    rows = np.sort(np.random.default_rng(9).choice(spec.N, size=16, replace=False))
    w_rows = w[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16)
    for B in (1, 4):
        x = synth.gen_x_np(B, spec.K, 6200 + B)
        y = W.gemv(c, dev(x)).cpu().numpy()[:, rows].astype(np.float64)
        y_ref = O.gemv(w_rows, x)
        assert np.abs(y - y_ref).max() <= GEMV_TOL * np.abs(y_ref).max()
    c.free()
