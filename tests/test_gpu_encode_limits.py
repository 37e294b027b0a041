"""Encoder at the edge of its histogram counters, on the GPU.

hist_kernel counts into 16-bit halves; the grid is sized so that no half can
wrap even when every element of a tensor has one symbol.  The hardest cases
are constant tensors whose block count sits at that bound: a small tensor in
a batch dominated by a much larger one (its share of the grid drops to the
bound) and a tensor of more than 1.9e9 elements encoded alone.  The small
tensor's container must equal the oracle's byte for byte; the large ones
must round-trip and carry the table and escape count the oracle gives for
the same constant on a small tensor.
"""
import numpy as np
import pytest

from oracle import wcomp_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def W():
    from decode_gemv_sign_gb300 import build, wcomp

    build.build()
    wcomp.lib()
    return wcomp


def dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("value", [0x0000, 0x3F80])
def test_constant_tensor_beside_a_huge_one(W, value):
    """512 x 8191 constant elements in a batch with 2.1e9 others: the grid gives the small
    tensor the fewest blocks the counter bound allows (the old bound wrapped here)."""
    small = np.full((512, 8191), value, dtype=np.uint16)
    big_n = 2_100_000_000
    g = torch.Generator(device="cuda")
    g.manual_seed(91)
    big = (torch.randn(big_n, generator=g, device="cuda") * 0.02).to(torch.bfloat16).view(torch.int16)
    big = big.reshape(50_000, 42_000)
    for scheme in O.SCHEMES:
        cs = W.encode_batched([dev(small), big], [scheme, scheme])
        ref = O.encode(small, scheme)
        inf = cs[0].info()
        assert inf["n_escapes"] == ref.E == 0
        assert inf["table"] == [int(t) for t in ref.table]
        assert W.serialize(cs[0]) == O.serialize(ref)
        out = W.decode(cs[1])
        assert torch.equal(out.view(-1), big.view(-1))
        del out
        for c in cs:
            c.free()
    del big
    torch.cuda.empty_cache()


def test_constant_tensor_alone_at_the_bound(W):
    """A constant tensor of 2^31 elements alone: its block count is set by the counter
    bound, not by the SM count."""
    n = 1 << 31
    value = 0xBC00
    w = torch.full((1 << 16, 1 << 15), value - 65536, dtype=torch.int16, device="cuda")
    small = np.full((4, 64), value, dtype=np.uint16)
    for scheme in O.SCHEMES:
        ref = O.encode(small, scheme)  # the table of a constant tensor does not depend on its size
        c = W.encode(w, scheme)
        inf = c.info()
        assert inf["n"] == n
        assert inf["n_escapes"] == 0
        assert inf["table"] == [int(t) for t in ref.table]
        out = W.decode(c)
        assert torch.equal(out, w)
        del out
        c.free()
    del w
    torch.cuda.empty_cache()
