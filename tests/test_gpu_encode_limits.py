"""Encoder at the edge of its histogram counters, on the GPU.

hist_kernel counts into 16-bit halves; the grid is sized so that no half can
wrap even when every element of a tensor has one symbol.  The hardest case
is a constant tensor whose block count sits at that bound: a small tensor in
a batch dominated by much larger ones (its share of the grid drops to the
bound).  A constant tensor of 2^31 elements encoded alone is the other large
case.  The small
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


def hist_blocks(W, ns):
    import ctypes

    arr = (ctypes.c_uint64 * len(ns))(*ns)
    out = (ctypes.c_uint32 * len(ns))()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert W.lib().wcomp_encode_hist_grid(arr, len(ns), sms, out) == W.OK
    return list(out)


@pytest.mark.parametrize("value", [0x0000, 0x3F80])
def test_constant_tensor_beside_huge_ones(W, value):
    """512 x 8191 constant elements in a batch with 5.2e9 others: the grid gives the small
    tensor the fewest blocks the counter bound allows (the old bound wrapped here)."""
    small = np.full((512, 8191), value, dtype=np.uint16)
    shape = (52_000, 50_000)  # two of these: 5.2e9 elements
    need = -(-(-(-small.size // 8)) // (1023 * 256))
    assert hist_blocks(W, [small.size, shape[0] * shape[1], shape[0] * shape[1]])[0] == need == 3
    g = torch.Generator(device="cuda")
    g.manual_seed(91)
    bigs = []
    for _ in range(2):
        b = torch.empty(shape, dtype=torch.int16, device="cuda")
        for r in range(0, shape[0], 4000):  # drawn in slices to bound the float32 temporary
            rows = min(4000, shape[0] - r)
            b[r:r + rows] = (torch.randn(rows, shape[1], generator=g, device="cuda") * 0.02).to(torch.bfloat16).view(torch.int16)
        bigs.append(b)
    for scheme in O.SCHEMES:
        cs = W.encode_batched([dev(small)] + bigs, [scheme] * 3)
        ref = O.encode(small, scheme)
        inf = cs[0].info()
        assert inf["n_escapes"] == ref.E == 0
        assert inf["table"] == [int(t) for t in ref.table]
        assert W.serialize(cs[0]) == O.serialize(ref)
        for c, b in zip(cs[1:], bigs):
            out = W.decode(c)
            assert torch.equal(out.view(-1), b.view(-1))
            del out
        for c in cs:
            c.free()
    del bigs
    torch.cuda.empty_cache()


def test_constant_tensor_of_2_31_elements_alone(W):
    """A constant tensor of 2^31 elements alone (every counter half of its blocks fed by one
    symbol) carries the oracle's table and escape count and round-trips."""
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
