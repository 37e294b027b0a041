"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Bars: container bytes and decoded BF16 bit-exact; GEMV within
max|y - y_oracle| <= 1e-4 * max|y_oracle| (fp32 accumulation against the
float64 oracle); one-hot x reproduces the weight column exactly.
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


def dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


GUARD = 4096  # elements of pattern on each side of a guarded output


class Guarded:
    """A device output with guard regions before and after it, filled with a
    known bit pattern: a store past either end of the output (which a kernel
    writing exactly-sized buffers could otherwise make unseen) changes them."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.n = n
        word = torch.int16 if dtype == torch.int16 else torch.int32
        self.pattern = 0x5A5A if word == torch.int16 else 0x7FBADBAD
        self.raw = torch.full((n + 2 * GUARD,), self.pattern, dtype=word, device="cuda")
        self.out = self.raw.view(dtype)[GUARD:GUARD + n].view(*shape)

    def check(self):
        head, tail = self.raw[:GUARD], self.raw[GUARD + self.n:]
        assert bool((head == self.pattern).all()) and bool((tail == self.pattern).all()), "guard region overwritten"


def check_gemv(y_gpu, y_ref):
    y = y_gpu.cpu().numpy().astype(np.float64)
    scale = np.abs(y_ref).max()
    err = np.abs(y - y_ref).max()
    assert err <= GEMV_TOL * scale, (err, scale)


CASES = {
    "fixture5x200": lambda: synth.gen_weights_np(synth.WeightSpec("g", 5, 200, "t4", 0.02, 0.05, "normal", 100.0, seed=77)),
    "all65536": lambda: np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256),
    "shuffled65536": lambda: np.random.default_rng(3).permutation(np.arange(65536, dtype=np.uint32).astype(np.uint16)).reshape(128, 512),
    "n1": lambda: np.array([[0x3F80]], dtype=np.uint16),
    "n3": lambda: np.array([[0x3F80, 0xFF80, 0x0001]], dtype=np.uint16),
    "n31": lambda: np.random.default_rng(31).integers(0, 65536, size=(1, 31)).astype(np.uint16),
    "n33": lambda: np.random.default_rng(33).integers(0, 65536, size=(3, 11)).astype(np.uint16),
    "n8191": lambda: np.random.default_rng(8191).integers(0, 65536, size=(1, 8191)).astype(np.uint16),
    "n8193": lambda: synth.gen_weights_np(synth.WeightSpec("r", 1, 8193, "normal", 0.02, 0.01, "normal", 1.0, seed=8)),
    "ragged7x301": lambda: synth.gen_weights_np(synth.WeightSpec("r", 7, 301, "t4", 0.02, 0.01, "normal", 1.0, seed=11)),
    "tiles_40000x3": lambda: synth.gen_weights_np(synth.WeightSpec("r", 3, 40000, "t4", 0.02, 0.01, "normal", 1.0, seed=12)),
    "specials": lambda: np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x807F] * 100, dtype=np.uint16).reshape(8, 100),
    "one_symbol": lambda: np.full((64, 64), 0x3C11, dtype=np.uint16),
    "w1024": lambda: synth.gen_weights_np(synth.workload_small()[0]),
}


@pytest.mark.parametrize("scheme", O.SCHEMES)
@pytest.mark.parametrize("case", list(CASES))
def test_container_and_decode_bit_exact(W, case, scheme):
    w = CASES[case]()
    ref = O.encode(w, scheme)
    c = W.encode(dev(w), scheme)
    inf = c.info()
    assert inf["n_escapes"] == ref.E
    assert inf["table"] == [int(t) for t in ref.table]
    assert W.serialize(c) == O.serialize(ref)
    compact = O.serialize_compact(ref)
    assert W.serialize(c, compact=True) == compact
    assert inf["serialized_compact_bytes"] == len(compact)
    g = Guarded(w.shape, torch.int16)
    out = W.decode(c, g.out)
    assert np.array_equal(host(out).reshape(w.shape), w)
    g.check()
    c.free()
    # the compact bytes load back into the same device container
    c2 = W.deserialize(compact)
    assert W.serialize(c2) == O.serialize(ref)
    assert np.array_equal(host(W.decode(c2)).reshape(w.shape), w)
    c2.free()


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_unaligned_pointers(W, scheme):
    w = synth.gen_weights_np(synth.WeightSpec("u", 9, 4096, "t4", 0.02, 0.01, "normal", 1.0, seed=21))
    flat = np.concatenate([np.zeros(1, np.uint16), w.reshape(-1), np.zeros(1, np.uint16)])
    big = dev(flat)
    c = W.encode(big[1:1 + w.size].view(9, 4096), scheme)  # input offset by 2 bytes
    assert W.serialize(c) == O.serialize(O.encode(w, scheme))
    out = torch.zeros(w.size + 1, dtype=torch.int16, device="cuda")
    W.decode(c, out[1:])  # output offset by 2 bytes
    assert np.array_equal(host(out[1:]).reshape(w.shape), w)
    xb = synth.gen_x_np(2, 4096, 5)
    xf = dev(np.concatenate([np.zeros(1, np.uint16), xb.reshape(-1)]))
    y = W.gemv(c, xf[1:].view(2, 4096))  # x offset: element path
    check_gemv(y, O.gemv(w, xb))
    c.free()


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_deserialize_roundtrip_on_gpu(W, scheme):
    w = synth.gen_weights_np(synth.WeightSpec("d", 33, 1024, "t4", 0.02, 0.01, "normal", 1.0, seed=13))
    buf = O.serialize(O.encode(w, scheme))
    c = W.deserialize(buf)
    assert np.array_equal(host(W.decode(c)).reshape(w.shape), w)
    assert W.serialize(c) == buf
    bad = bytearray(buf)
    bad[200] ^= 1
    with pytest.raises(W.CorruptContainer):
        W.deserialize(bytes(bad))


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_compact_form_on_gpu(W, scheme):
    """Library-made compact bytes load back (oracle and library agree both ways),
    and a container loaded from them runs the fused GEMV like the original."""
    spec = synth.WeightSpec("d", 64, 2048, "t4", 0.02, 0.01, "normal", 1.0, seed=14)
    w = synth.gen_weights_np(spec)
    c = W.encode(dev(w), scheme)
    buf = W.serialize(c, compact=True)
    back = O.deserialize(buf)
    assert O.serialize(back) == W.serialize(c)
    c2 = W.deserialize(buf)
    x = synth.gen_x_np(4, spec.K, 15)
    assert torch.equal(W.gemv(c2, dev(x)), W.gemv(c, dev(x)))
    bad = bytearray(buf)
    bad[300] ^= 1
    with pytest.raises(W.CorruptContainer):
        W.deserialize(bytes(bad))
    c.free()
    c2.free()


@pytest.mark.parametrize("scheme", O.SCHEMES)
@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 8, 12, 16])
def test_gemv_matches_oracle(W, scheme, B):
    spec = synth.WeightSpec("g", 300, 2048, "t4", 0.02, 0.005, "normal", 1.0, seed=100 + B)
    w = synth.gen_weights_np(spec)
    x = synth.gen_x_np(B, spec.K, 200 + B)
    c = W.encode(dev(w), scheme)
    g = Guarded((B, spec.N), torch.float32)
    y = W.gemv(c, dev(x), g.out)
    check_gemv(y, O.gemv(w, x))
    g.check()
    # deterministic: same bits on a second call
    y2 = W.gemv(c, dev(x))
    assert torch.equal(y, y2)
    W.device_check()  # no kernel reported a timed-out wait
    c.free()


@pytest.mark.parametrize("B", [3, 4, 6, 8])
def test_gemv_k15_walk_offsets(W, B):
    """K15 at B = 3..8 walks each warp's k-blocks from a per-unit offset
    (wrapping) where a warp has at least 16 of them: with 17 per warp
    (K = 17408) the first units start at offsets 0, 7, 14, 4, 11; with 41
    (K = 41984) and 96 rows at 0, 7, .., 35; with 5 (K = 5120) in order.
    Every sum must still cover each k-block once, and the result must not
    depend on the call."""
    for seed, (N, K) in enumerate([(80, 17408), (96, 41984), (80, 5120)]):
        spec = synth.WeightSpec("r", N, K, "t4", 0.02, 0.005, "normal", 1.0, seed=500 + 10 * B + seed)
        w = synth.gen_weights_np(spec)
        x = synth.gen_x_np(B, K, 600 + 10 * B + seed)
        c = W.encode(dev(w), 1)
        g = Guarded((B, N), torch.float32)
        y = W.gemv(c, dev(x), g.out)
        check_gemv(y, O.gemv(w, x))
        g.check()
        assert torch.equal(y, W.gemv(c, dev(x)))
        W.device_check()
        c.free()


@pytest.mark.parametrize("B", [9, 16])
def test_plain_gemv_walk_offsets(W, B):
    """The plain GEMV above B = 8 walks each warp's k-blocks from the same
    per-unit offsets as K15 at B = 3..8 (17 and 41 k-blocks a warp here)."""
    for seed, (N, K) in enumerate([(80, 17408), (96, 41984)]):
        spec = synth.WeightSpec("p", N, K, "t4", 0.02, 0.005, "normal", 1.0, seed=700 + 10 * B + seed)
        w = synth.gen_weights_np(spec)
        x = synth.gen_x_np(B, K, 800 + 10 * B + seed)
        g = Guarded((B, N), torch.float32)
        y = W.gemv_bf16(dev(w), dev(x), g.out)
        check_gemv(y, O.gemv(w, x))
        g.check()
        assert torch.equal(y, W.gemv_bf16(dev(w), dev(x)))
        W.device_check()


@pytest.mark.parametrize("scheme", O.SCHEMES + (2,))
@pytest.mark.parametrize("shape", [(37, 96), (64, 160), (9, 2080), (8, 32), (130, 1056)])
@pytest.mark.parametrize("B", [1, 2, 4, 8, 9, 16])
def test_gemv_partial_blocks(W, scheme, shape, B):
    """K not a multiple of the 1024-element chunk or the 128-element k-block
    (partial last blocks, lanes past K, warps with no k-block at all when K <
    1024) and N not a multiple of 8 (a partial 8-row unit), for both GEMV
    kernels; scheme 2 is the plain BF16 GEMV."""
    N, K = shape
    spec = synth.WeightSpec("p", N, K, "t4", 0.02, 0.01, "normal", 1.0, seed=31 * N + K)
    w = synth.gen_weights_np(spec)
    x = synth.gen_x_np(B, K, 17 * B + K)
    g = Guarded((B, N), torch.float32)
    if scheme == 2:
        y = W.gemv_bf16(dev(w), dev(x), g.out)
    else:
        c = W.encode(dev(w), scheme)
        y = W.gemv(c, dev(x), g.out)
        c.free()
    check_gemv(y, O.gemv(w, x))
    g.check()


@pytest.mark.parametrize("scheme", O.SCHEMES)
@pytest.mark.parametrize("B", [1, 4, 16])
def test_gemv_ragged_k_element_path(W, scheme, B):
    spec = synth.WeightSpec("g", 37, 1000, "t4", 0.02, 0.01, "normal", 1.0, seed=300 + B)
    w = synth.gen_weights_np(spec)
    x = synth.gen_x_np(B, spec.K, 301)
    c = W.encode(dev(w), scheme)
    check_gemv(W.gemv(c, dev(x)), O.gemv(w, x))
    c.free()


def _escapes_on_boundaries(N, K, scheme):
    """W[N, K] of 15 common symbols in turn (magnitudes 2^-15 .. 2), with a
    rare symbol (2.0 .. 4.0) on every row start and row end and on both sides
    of every 8192-element tile boundary; the raw bits count up."""
    n = N * K
    i = np.arange(n)
    mask = 0xFF if scheme == O.BYTESPLIT else 0x7F
    common = np.array([0x3C, 0x3D, 0x3E, 0x3F, 0xBC, 0xBD, 0xBE, 0xBF, 0x3B, 0xBB, 0x3A, 0xBA, 0x39, 0xB9, 0x38])
    w = ((common[i % 15] << 8) | (i & mask)).astype(np.uint16)
    spots = set()
    for r in range(N):
        spots |= {r * K, r * K + K - 1}
    for t in range(1, -(-n // O.TILE)):
        spots |= {t * O.TILE - 1, t * O.TILE}
    spots = sorted(spots)
    w[spots] = 0x4000 | (i[spots] & mask)
    return w.reshape(N, K), spots


@pytest.mark.parametrize("scheme", O.SCHEMES)
@pytest.mark.parametrize("shape", [(3, 8197), (6, 8192), (40, 1024)])
def test_escapes_on_row_and_tile_boundaries(W, scheme, shape):
    """Escapes exactly where rows and tiles begin and end: containers and
    decode bit-exact, GEMV within tolerance for a ragged K (element path) and
    aligned K (FMA and tensor-core kernels)."""
    w, spots = _escapes_on_boundaries(*shape, scheme)
    ref = O.encode(w, scheme)
    assert ref.esc_pos.tolist() == spots
    c = W.encode(dev(w), scheme)
    assert W.serialize(c) == O.serialize(ref)
    assert W.serialize(c, compact=True) == O.serialize_compact(ref)
    gd = Guarded(w.shape, torch.int16)
    assert np.array_equal(host(W.decode(c, gd.out)).reshape(w.shape), w)
    gd.check()
    for B in (1, 4, 16):
        x = synth.gen_x_np(B, shape[1], 40 + B)
        gy = Guarded((B, shape[0]), torch.float32)
        check_gemv(W.gemv(c, dev(x), gy.out), O.gemv(w, x))
        gy.check()
    c.free()


def _escapes_per_row(N, K, seed):
    """W[N, K] of common symbols with row r holding r % 11 escapes (rare
    exponents) at seeded columns, so that a row's first escape entry falls at
    every residue mod 4 of the stream and rows with 0..10 escapes alternate
    (each row's first and last groups of four entries are partial)."""
    rng = np.random.default_rng(seed)
    common = np.array([0x3C, 0x3D, 0x3E, 0x3F, 0xBC, 0xBD, 0xBE, 0xBF, 0x3B, 0xBB, 0x3A, 0xBA, 0x39, 0xB9, 0x38])
    hi = common[rng.integers(0, 15, size=(N, K))]
    lo = rng.integers(0, 128, size=(N, K))  # exponent bit 0 clear: 15 nine-bit symbols too
    w = ((hi << 8) | lo).astype(np.uint16)
    for r in range(N):
        cols = rng.choice(K, size=r % 11, replace=False)
        w[r, cols] = ((0x40 + rng.integers(0, 4, size=cols.size)) << 8 | rng.integers(0, 256, size=cols.size)).astype(np.uint16)
    return w


@pytest.mark.parametrize("scheme", O.SCHEMES)
@pytest.mark.parametrize("B", [1, 2, 3, 5, 8, 9, 16])
def test_gemv_escape_counts_per_row(W, scheme, B):
    """Rows with 0..10 escapes each, over several 16-row units and every
    alignment of a row's entries in the escape stream: the fused GEMV (single
    entries, aligned groups of four, transposed x) matches the oracle, and the
    output's guard regions stay intact."""
    N, K = 83, 2048
    w = _escapes_per_row(N, K, 900 + B)
    ref = O.encode(w, scheme)
    counts = np.bincount(np.asarray(ref.esc_pos) // K, minlength=N)
    assert counts.tolist() == [r % 11 for r in range(N)]
    x = synth.gen_x_np(B, K, 910 + B)
    c = W.encode(dev(w), scheme)
    g = Guarded((B, N), torch.float32)
    check_gemv(W.gemv(c, dev(x), g.out), O.gemv(w, x))
    g.check()
    W.device_check()
    c.free()


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_gemv_one_hot_exact_and_zero(W, scheme):
    spec = synth.WeightSpec("o", 64, 256, "normal", 0.02, 0.05, "normal", 1.0, seed=5)
    w = synth.gen_weights_np(spec)
    ref = O.encode(w, scheme)
    assert ref.E > 0
    c = W.encode(dev(w), scheme)
    ks = sorted(set([0, 1, 31, 32, 255] + [int(p) % spec.K for p in ref.esc_pos[:12]]))
    x = np.zeros((len(ks), spec.K), np.uint16)
    for i, k in enumerate(ks):
        x[i, k] = 0x3F80
    for b0 in range(0, len(ks), 16):
        xb = x[b0:b0 + 16]
        y = W.gemv(c, dev(xb)).cpu().numpy()
        for i in range(xb.shape[0]):
            col = (w[:, ks[b0 + i]].astype(np.uint32) << 16).view(np.float32)
            assert np.array_equal(y[i], col)
    y0 = W.gemv(c, torch.zeros((4, spec.K), dtype=torch.int16, device="cuda"))
    assert not y0.any()
    c.free()


@pytest.mark.parametrize("B", [1, 3, 4, 16])
def test_plain_bf16_gemv(W, B):
    spec = synth.WeightSpec("p", 257, 4096, "normal", 0.02, seed=7)
    w = synth.gen_weights_np(spec)
    x = synth.gen_x_np(B, spec.K, 8)
    check_gemv(W.gemv_bf16(dev(w), dev(x)), O.gemv(w, x))
    w2 = synth.gen_weights_np(synth.WeightSpec("p", 13, 1000, "normal", 0.02, seed=9))
    x2 = synth.gen_x_np(B, 1000, 10)
    check_gemv(W.gemv_bf16(dev(w2), dev(x2)), O.gemv(w2, x2))


def test_plain_batched(W):
    shapes = [(64, 1024), (33, 1000), (200, 2048), (5, 4096)]
    ws = [synth.gen_weights_np(synth.WeightSpec(f"q{i}", N, K, "normal", 0.02, seed=800 + i))
          for i, (N, K) in enumerate(shapes)]
    for B in (1, 4, 16):
        xs = [synth.gen_x_np(B, K, 900 + i) for i, (_, K) in enumerate(shapes)]
        ys = W.gemv_bf16_batched([dev(w) for w in ws], [dev(x) for x in xs])
        for w, x, y in zip(ws, xs, ys):
            check_gemv(y, O.gemv(w, x))


def test_batched_matches_single(W):
    specs = [synth.WeightSpec(f"b{i}", N, K, "t4", 0.02, 0.01, "normal", 1.0, seed=400 + i)
             for i, (N, K) in enumerate([(64, 1024), (200, 640), (33, 1000), (128, 2048), (1, 4096)])]
    ws = [synth.gen_weights_np(s) for s in specs]
    cs = [W.encode(dev(w), i % 2) for i, w in enumerate(ws)]
    gd = [Guarded(w.shape, torch.int16) for w in ws]
    outs = W.decode_batched(cs, [g.out for g in gd])
    for w, o, g in zip(ws, outs, gd):
        assert np.array_equal(host(o).reshape(w.shape), w)
        g.check()
    for B in (1, 4):
        xs = [synth.gen_x_np(B, s.K, 500 + i) for i, s in enumerate(specs)]
        gy = [Guarded((B, s.N), torch.float32) for s in specs]
        ys = W.gemv_batched(cs, [dev(x) for x in xs], [g.out for g in gy])
        for c, w, x, y, g in zip(cs, ws, xs, ys, gy):
            check_gemv(y, O.gemv(w, x))
            g.check()
            assert torch.equal(y, W.gemv(c, dev(x)))
    for c in cs:
        c.free()


def test_encode_batched_matches_single(W):
    specs = [synth.WeightSpec(f"e{i}", N, K, "t4", 0.02, 0.01, "normal", 1.0, seed=1000 + i)
             for i, (N, K) in enumerate([(64, 1024), (1, 31), (33, 1000), (128, 2048), (3, 40000), (7, 301)])]
    ws = [synth.gen_weights_np(s) for s in specs]
    schemes = [i % 2 for i in range(len(ws))]
    cs = W.encode_batched([dev(w) for w in ws], schemes)
    for w, c, sc in zip(ws, cs, schemes):
        assert W.serialize(c) == O.serialize(O.encode(w, sc))
    # more tensors than one launch carries, mixed schemes and shapes
    ws2 = [synth.gen_weights_np(synth.WeightSpec(f"f{i}", 8 + i, 256 + 32 * (i % 5), "normal", 0.02, 0.02,
                                                 "normal", 1.0, seed=1100 + i)) for i in range(75)]
    cs2 = W.encode_batched([dev(w) for w in ws2], [(i // 3) % 2 for i in range(75)])
    for i, (w, c) in enumerate(zip(ws2, cs2)):
        assert W.serialize(c) == O.serialize(O.encode(w, (i // 3) % 2))
        assert np.array_equal(host(W.decode(c)).reshape(w.shape), w)


def test_encode_batched_both_schemes_of_one_tensor(W):
    # the byte-split job folds the K15 histogram of the same tensor
    specs = [synth.WeightSpec(f"t{i}", N, K, "t4", 0.02, 0.01, "normal", 1.0, seed=1200 + i)
             for i, (N, K) in enumerate([(64, 1024), (3, 40000), (7, 301), (1, 31)])]
    ws = [synth.gen_weights_np(s) for s in specs]
    wd = [dev(w) for w in ws]
    cs = W.encode_batched([w for w in wd for _ in (0, 1)], [1, 0] * len(wd))
    for i, w in enumerate(ws):
        assert W.serialize(cs[2 * i]) == O.serialize(O.encode(w, 1))
        assert W.serialize(cs[2 * i + 1]) == O.serialize(O.encode(w, 0))
    w65 = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    d65 = dev(w65)
    c0, c1 = W.encode_batched([d65, d65], [0, 1])
    assert W.serialize(c0) == O.serialize(O.encode(w65, 0))
    assert W.serialize(c1) == O.serialize(O.encode(w65, 1))


def test_encode_twins_over_one_launch_and_unpaired(W):
    # 20 tensors in both schemes (20 byte-split/K15 pairs: more than one twin
    # launch carries), plus a third encode of one tensor that has no twin left
    specs = [synth.WeightSpec(f"p{i}", 8 + i, 512 + 32 * i, "normal", 0.02, 0.01, "normal", 1.0, seed=1300 + i)
             for i in range(20)]
    ws = [synth.gen_weights_np(s) for s in specs]
    wd = [dev(w) for w in ws]
    tensors = [w for w in wd for _ in (0, 1)] + [wd[3]]
    schemes = [0, 1] * len(wd) + [0]
    cs = W.encode_batched(tensors, schemes)
    for i, w in enumerate(ws):
        assert W.serialize(cs[2 * i]) == O.serialize(O.encode(w, 0))
        assert W.serialize(cs[2 * i + 1]) == O.serialize(O.encode(w, 1))
    assert W.serialize(cs[-1]) == O.serialize(O.encode(ws[3], 0))


def test_many_tensors_batch_over_limit(W):
    # more containers than one launch carries
    ws = [synth.gen_weights_np(synth.WeightSpec(f"m{i}", 16, 512, "normal", 0.02, 0.01, "normal", 1.0, seed=600 + i))
          for i in range(70)]
    cs = [W.encode(dev(w), i % 2) for i, w in enumerate(ws)]
    outs = W.decode_batched(cs)
    for w, o in zip(ws, outs):
        assert np.array_equal(host(o).reshape(w.shape), w)
    xs = [synth.gen_x_np(1, 512, 700 + i) for i in range(70)]
    ys = W.gemv_batched(cs, [dev(x) for x in xs])
    for w, x, y in zip(ws, xs, ys):
        check_gemv(y, O.gemv(w, x))


def test_argument_errors(W):
    w = dev(np.zeros((4, 64), np.uint16))
    c = W.encode(w, 0)
    with pytest.raises(W.WcompError):
        W.gemv(c, torch.zeros((17, 64), dtype=torch.int16, device="cuda"))
    with pytest.raises(ValueError):
        W.decode(c, torch.zeros(10, dtype=torch.int16, device="cuda"))
    c.free()
