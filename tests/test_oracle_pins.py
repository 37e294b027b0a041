"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Nothing here re-types an oracle formula and compares it with itself.  The
pins are: exact round trip (the pages' definition of lossless) by brute force
over every BF16 bit pattern; an independent per-element pure-Python reader
of the serialized bytes; hand-derived closed forms of the stream sizes and
bit positions; counting by brute force for the histogram and the table; the
accounting identities printed on the pages; and one-hot / zero / brute-force
dot products for the GEMV.
"""
import json
import os
import struct
import zlib

import numpy as np
import pytest

from decode_gemv_sign_gb300 import synth
from oracle import wcomp_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
PAGES = json.load(open(os.path.join(HERE, "golden", "pages_figures.json")))


# ---------------------------------------------------------------------------
# An independent reader of serialized containers, one element at a time.
# ---------------------------------------------------------------------------
def _pad(x):
    return (x + 31) // 32 * 32


def read_element_pure(buf: bytes, i: int) -> int:
    """Rebuild weight i from the serialized bytes with plain integer code."""
    scheme = buf[6]
    N, K, E = struct.unpack_from("<qqQ", buf, 8)
    n = N * K
    table = struct.unpack_from("<15H", buf, 40)
    p = 96
    codes_off = p
    p += _pad((n + 1) // 2)
    groups = (n + 31) // 32
    if scheme == 0:
        raw_off = p
        p += _pad(n)
    else:
        a_off = p
        p += _pad(16 * groups)
        b_off = p
        p += _pad(8 * groups)
        c_off = p
        p += _pad(4 * groups)
    n_tiles = (n + 8191) // 8192
    p += _pad(4 * (n_tiles + 1))
    p += _pad(4 * (N + 1))
    pos_off = p
    p += _pad(4 * E)
    val_off = p
    byte = buf[codes_off + i // 2]
    code = (byte >> 4) if i % 2 else (byte & 15)
    if scheme == 0:
        low = buf[raw_off + i]
    else:
        g, e = divmod(i, 32)
        # byte j of the group's 28 mantissa bytes: 16 in section A, 8 in B, 4 in C
        def mbyte(j):
            if j < 16:
                return buf[a_off + 16 * g + j]
            if j < 24:
                return buf[b_off + 8 * g + j - 16]
            return buf[c_off + 4 * g + j - 24]
        if e < 28:
            low = mbyte(e) & 0x7F
        else:
            low = sum(((mbyte(4 * b + e - 28) >> 7) & 1) << b for b in range(7))
    if code != 15:
        sym = table[code]
        return (sym << 8) | low if scheme == 0 else (sym << 7) | low
    # linear search of the escape stream
    for e in range(E):
        if struct.unpack_from("<I", buf, pos_off + 4 * e)[0] == i:
            if scheme == 0:
                return (buf[val_off + e] << 8) | low
            return struct.unpack_from("<H", buf, val_off + 2 * e)[0]
    raise AssertionError("escape code without an escape entry")


def _roundtrip(w, scheme, N=None, K=None):
    c = O.encode(w, scheme, N, K)
    buf = O.serialize(c)
    back = O.decode(O.deserialize(buf))
    assert np.array_equal(back.reshape(-1), np.asarray(w, np.uint16).reshape(-1))
    return c, buf


# ---------------------------------------------------------------------------
# Exactness: every BF16 bit pattern.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_all_65536_patterns_roundtrip(scheme):
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    c, buf = _roundtrip(w.reshape(256, 256), scheme)
    # every symbol value appears equally often: ties broken by symbol value
    assert list(c.table) == list(range(15))
    # everything whose symbol is not among the first 15 escapes
    per_sym = 65536 // O.NBINS[scheme]
    assert c.E == 65536 - 15 * per_sym
    rng = np.random.default_rng(7)
    for _ in range(2):
        ws = rng.permutation(w).astype(np.uint16)
        _roundtrip(ws.reshape(128, 512), scheme)
    # the independent reader agrees on a sample of elements, including escapes
    for i in list(range(0, 65536, 997)) + [c.esc_pos[0], c.esc_pos[-1], 65535]:
        assert read_element_pure(buf, int(i)) == int(w[i])


@pytest.mark.parametrize("scheme", O.SCHEMES)
@pytest.mark.parametrize("n", [1, 2, 3, 31, 32, 33, 8191, 8192, 8193, 65537])
def test_ragged_sizes_roundtrip(scheme, n):
    rng = np.random.default_rng(n)
    w = rng.integers(0, 65536, size=n).astype(np.uint16)
    c, buf = _roundtrip(w, scheme)
    for i in sorted(set([0, n - 1, n // 2] + list(rng.integers(0, n, size=20)))):
        assert read_element_pure(buf, int(i)) == int(w[i])


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_special_values_roundtrip(scheme):
    specials = [0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x807F, 0x3F80, 0xBF80, 0x7F7F]
    w = np.array(specials * 37, dtype=np.uint16)
    _roundtrip(w, scheme)


# ---------------------------------------------------------------------------
# Histogram and table by brute-force counting.
# ---------------------------------------------------------------------------
def _brute_table(w, scheme):
    counts = {}
    for v in np.asarray(w).reshape(-1).tolist():
        s = v >> 8 if scheme == 0 else v >> 7
        counts[s] = counts.get(s, 0) + 1
    nb = 256 if scheme == 0 else 512
    ranked = sorted(range(nb), key=lambda s: (-counts.get(s, 0), s))
    return ranked[:15], counts


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_histogram_and_table_brute_force(scheme):
    w = synth.gen_weights_np(synth.WeightSpec("t", 7, 301, "t4", 0.02, 0.01, "normal", 1.0, seed=11))
    sym, _ = O.split_symbols(w, scheme)
    h = O.histogram(sym, scheme)
    table, counts = _brute_table(w, scheme)
    assert h.sum() == w.size
    # one bin per possible symbol: 2^8 high bytes, 2^9 sign+exponent values
    assert h.size == (256 if scheme == 0 else 512)
    assert all(h[s] == counts.get(s, 0) for s in range(h.size))
    assert list(O.select_table(h)) == table


@pytest.mark.parametrize("scheme", O.SCHEMES)
@pytest.mark.parametrize("distinct", [1, 15, 16, 17])
def test_distinct_symbol_counts(scheme, distinct):
    shift = 8 if scheme == 0 else 7
    rng = np.random.default_rng(distinct)
    # symbol s_j occurs 100 + j times (so the least frequent escape first)
    syms = [(37 + 5 * j) % (1 << (16 - shift)) for j in range(distinct)]
    vals = []
    for j, s in enumerate(syms):
        for _ in range(100 + (distinct - j)):
            vals.append((s << shift) | int(rng.integers(0, 1 << shift)))
    w = rng.permutation(np.array(vals, dtype=np.uint16))
    c, _ = _roundtrip(w, scheme)
    expect_esc = sum(100 + (distinct - j) for j in range(15, distinct))
    assert c.E == expect_esc
    # the table starts with the most frequent symbols; unseen symbols fill it ascending
    seen = syms[: min(distinct, 15)]
    assert list(c.table[: len(seen)]) == seen
    if distinct < 15:
        fill = [s for s in range(1 << (16 - shift)) if s not in syms][: 15 - distinct]
        assert list(c.table[distinct:]) == fill


def test_all_escape_except_table():
    # 400 distinct high bytes, each twice: 15 coded, the rest escapes
    w = np.array([(s << 8) | 0x5A for s in range(256)] * 2, dtype=np.uint16)
    c, _ = _roundtrip(w, O.BYTESPLIT)
    assert c.E == 2 * (256 - 15)


# ---------------------------------------------------------------------------
# Layout at the bit level: hand-derived positions.
# ---------------------------------------------------------------------------
def test_nibble_order_fixture():
    # table from counts: symbol 0x3C most frequent, then 0xBC, then 0x3D
    w = np.array([0x3C01] * 5 + [0xBC02] * 4 + [0x3D03] * 3, dtype=np.uint16)
    c = O.encode(w, O.BYTESPLIT)
    assert list(c.table[:3]) == [0x3C, 0xBC, 0x3D]
    # element 0 -> code 0 (low nibble), element 5 -> code 1 -> byte 2 high nibble
    assert c.codes[2] == 0x10  # elements 4 (code 0) and 5 (code 1)
    assert c.codes[4] == 0x21  # elements 8 (code 1) and 9 (code 2)
    assert bytes(c.raw[:3]) == b"\x01\x01\x01"


def test_k15_plane_bit_positions():
    # group 0: element 13 (a head element) has mantissa 0b1011011, element 30
    # (tail element 2) has 0b1000101; group 1: element 32 + 5 = 0b1000001,
    # tail element 32 + 31 (tail 3) = 0b0000011
    m = np.zeros(64, dtype=np.uint32)
    m[13] = 0b1011011
    m[30] = 0b1000101
    m[32 + 5] = 0b1000001
    m[32 + 31] = 0b0000011
    pa, pb, pc = O.pack_k15_planes(m)
    assert pa.size == 32 and pb.size == 16 and pc.size == 8  # 16 + 8 + 4 bytes per group
    mb0 = np.concatenate([pa[:16], pb[:8], pc[:4]])
    mb1 = np.concatenate([pa[16:], pb[8:], pc[4:]])
    # head element 13: byte 13, bits 0..6 (plane A, word 3, byte lane 1)
    expect0 = np.zeros(28, dtype=np.uint8)
    expect0[13] = 0b1011011
    # tail element 30 = 28 + 2: bit b in bit 7 of byte 4 b + 2; its bits 0, 2 and 6 are set
    for b in (0, 2, 6):
        expect0[4 * b + 2] |= 0x80
    assert np.array_equal(mb0, expect0)
    expect1 = np.zeros(28, dtype=np.uint8)
    expect1[5] = 0b1000001
    for b in (0, 1):  # tail element 3 of group 1 (element 63): bits 0 and 1
        expect1[4 * b + 3] |= 0x80
    assert np.array_equal(mb1, expect1)
    # the three sections as little-endian words: byte 13 is lane 1 of word 3 of plane A
    a = np.frombuffer(pa.tobytes(), "<u4")
    assert a[3] == 0b1011011 << 8 and a[1] == 0
    assert a[0] == 0x80 << 16 and a[2] == 0x80 << 16  # bits 0 and 2 of element 30 (lane 2 of words 0 and 2)
    cc = np.frombuffer(pc.tobytes(), "<u4")
    assert cc[0] == 0x80 << 16  # bit 6 of element 30: byte 26 = plane C byte 2
    back = O.unpack_k15_planes(pa, pb, pc, 64)
    assert np.array_equal(back, m)


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_serialized_size_closed_form(scheme):
    w = synth.gen_weights_np(synth.workload_small()[0])
    c = O.encode(w, scheme)
    buf = O.serialize(c)
    E = c.E
    if scheme == 0:
        # header 96, codes 524288, raw 1048576, tile index 129*4=516->544,
        # row index 1025*4=4100->4128, positions 4E, values E (each padded to 32)
        expect = 96 + 524288 + 1048576 + 544 + 4128 + _pad(4 * E) + _pad(E)
    else:
        # 32768 groups: planes 524288 + 262144 + 131072; values 2E
        expect = 96 + 524288 + 524288 + 262144 + 131072 + 544 + 4128 + _pad(4 * E) + _pad(2 * E)
    assert len(buf) == expect
    assert O.serialized_len(scheme, c.N, c.K, E) == expect
    # checksums are standard CRC-32 values over header / payload
    assert struct.unpack_from("<I", buf, 92)[0] == zlib.crc32(buf[:92])


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_escape_stream_and_indexes(scheme):
    w = synth.gen_weights_np(synth.WeightSpec("t", 9, 3000, "normal", 0.02, 0.02, "normal", 1.0, seed=3))
    c = O.encode(w, scheme)
    wf = w.reshape(-1).astype(np.int64)
    codes = O.unpack_codes(c.codes, c.n)
    # positions strictly ascending, exactly the elements coded 15
    assert np.all(np.diff(c.esc_pos.astype(np.int64)) > 0)
    assert np.array_equal(np.flatnonzero(codes == 15), c.esc_pos)
    shift = 8 if scheme == 0 else 7
    for e in range(0, c.E, max(1, c.E // 50)):
        p = int(c.esc_pos[e])
        assert (wf[p] >> shift) not in set(int(t) for t in c.table)
        if scheme == 0:
            assert int(c.esc_val[e]) == wf[p] >> 8
        else:
            assert int(c.esc_val[e]) == wf[p]
    # index entries count escapes below each boundary (brute force)
    for t in range(c.n_tiles + 1):
        assert c.tile_index[t] == sum(1 for p in c.esc_pos if p < t * O.TILE)
    for r in range(c.N + 1):
        assert c.row_index[r] == sum(1 for p in c.esc_pos if p < r * c.K)


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_indexes_with_escapes_on_boundaries(scheme):
    # 3 rows of K = 8192 + 5: escapes placed exactly on row starts, on tile
    # boundaries (multiples of 8192), on the element before each, and last.
    N, K = 3, 8197
    n = N * K
    shift = 8 if scheme == 0 else 7
    i = np.arange(n)
    # 15 common symbols in turn fill the table; the raw bits count up
    w = (((0x30 + i % 15) << 8) | (i & ((1 << shift) - 1))).astype(np.uint16)
    spots = [0, 8191, 8192, K - 1, K, 16383, 16384, 2 * K - 1, 2 * K, 24575, 24576, n - 1]
    w[spots] = 0x7F00  # a symbol seen only at these spots
    c = O.encode(w, scheme, N, K)
    assert c.E == len(spots) and c.esc_pos.tolist() == spots
    # entry j counts escapes strictly below boundary j
    assert c.tile_index.tolist() == [sum(p < t * 8192 for p in spots) for t in range(c.n_tiles + 1)]
    assert c.row_index.tolist() == [sum(p < r * K for p in spots) for r in range(N + 1)]
    assert c.row_index.tolist() == [0, 4, 8, len(spots)]
    # row 1 starts with an escape and row 0 ends with one: both stay in their rows
    assert np.array_equal(O.decode_rows(c, np.array([1])), w.reshape(N, K)[[1]])


# ---------------------------------------------------------------------------
# Corruption is detected.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_corruption_detected(scheme):
    w = synth.gen_weights_np(synth.WeightSpec("t", 16, 1024, "normal", 0.02, 0.01, "normal", 1.0, seed=5))
    buf = bytearray(O.serialize(O.encode(w, scheme)))
    O.deserialize(bytes(buf))
    rng = np.random.default_rng(0)
    for off in [0, 5, 9, 40, 80, 95] + list(rng.integers(96, len(buf), size=12)):
        bad = bytearray(buf)
        bad[off] ^= 0x10
        with pytest.raises(O.CorruptContainer):
            O.deserialize(bytes(bad))
    with pytest.raises(O.CorruptContainer):
        O.deserialize(bytes(buf[:-16]))
    with pytest.raises(O.CorruptContainer):
        O.deserialize(bytes(buf[:50]))


# ---------------------------------------------------------------------------
# Accounting against the pages' printed figures.
# ---------------------------------------------------------------------------
def test_accounting_identities_from_pages():
    bs = PAGES["bytesplit_bits_per_weight"]["value"]
    k15 = PAGES["k15_bits_per_weight"]["value"]
    # 16 * (1 - r): the pages print bpw and percentage rounded independently
    assert abs(O.reduction_pct(bs) - PAGES["bytesplit_reduction_pct"]["value"]) < 0.005
    assert abs(O.reduction_pct(k15) - PAGES["k15_reduction_pct"]["value"]) < 0.005
    before = PAGES["checkpoint_gib_before"]["value"]
    after = PAGES["checkpoint_gib_after_k15"]["value"]
    assert abs(before * k15 / 16 - after) < 0.02
    assert abs((before - after) - PAGES["checkpoint_gib_saved"]["value"]) < 0.5
    assert abs(before * 2**30 / 2 / 1e9 - PAGES["model_params_billions"]["value"]) < 1
    # 4 code bits + 8 (byte-split) or 7 (K15) raw bits is where both figures start
    assert int(bs) == 4 + 8 and int(k15) == 4 + 7


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_accounting_no_escapes_exact(scheme):
    # 3 distinct symbols -> E = 0: bits = 4 + raw + 15 table symbols
    w = np.array([0x3C00, 0x3C80, 0xBC11] * 1000, dtype=np.uint16)
    c = O.encode(w, scheme)
    assert c.E == 0
    raw, symb = (8, 8) if scheme == 0 else (7, 9)
    assert O.entropy_bpw(scheme, c.n, 0) == 4 + raw + 15 * symb / 3000


def test_accounting_on_gaussian_weights_matches_pages():
    # N(0, 0.02) BF16 weights: the pages' 12.005 (byte-split) and 11.173 (K15)
    spec = synth.WeightSpec("g", 1024, 4096, "normal", 0.02, seed=123)
    w = synth.gen_weights_np(spec)
    c0 = O.encode(w, O.BYTESPLIT)
    c1 = O.encode(w, O.K15)
    assert abs(O.entropy_bpw(O.BYTESPLIT, c0.n, c0.E) - PAGES["bytesplit_bits_per_weight"]["value"]) < 0.01
    assert abs(O.entropy_bpw(O.K15, c1.n, c1.E) - PAGES["k15_bits_per_weight"]["value"]) < 0.03


# ---------------------------------------------------------------------------
# GEMV.
# ---------------------------------------------------------------------------
def _f(b):
    return struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]


def test_gemv_brute_force_tiny():
    rng = np.random.default_rng(1)
    W = synth.f32_to_bf16_bits(rng.standard_normal((3, 5)).astype(np.float32))
    X = synth.f32_to_bf16_bits(rng.standard_normal((2, 5)).astype(np.float32))
    y = O.gemv(W, X)
    for b in range(2):
        for r in range(3):
            ref = sum(_f(X[b, k]) * _f(W[r, k]) for k in range(5))
            assert abs(y[b, r] - ref) <= 1e-15 * max(1.0, abs(ref))


def test_gemv_is_exact_where_fp32_accumulation_is_not():
    # 1 + 2^-30 needs 31 significant bits: exact in fp64, rounded to 1 by any
    # fp32 sum in any order.  Row 2: 1 + 2^-30 - 1 = 2^-30 exactly.
    W = np.array([[0x3F80, 0x3080, 0x0000], [0x3F80, 0x3080, 0xBF80]], np.uint16)  # 1, 2^-30, 0 / -1
    X = np.array([[0x3F80, 0x3F80, 0x3F80]], np.uint16)
    assert _f(0x3080) == 2.0 ** -30
    y = O.gemv(W, X)
    assert y[0, 0] == 1.0 + 2.0 ** -30
    assert y[0, 1] == 2.0 ** -30


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_gemv_one_hot_and_zero(scheme):
    w = synth.gen_weights_np(synth.WeightSpec("t", 33, 96, "normal", 0.02, 0.05, "normal", 1.0, seed=9))
    c = O.encode(w, scheme)
    assert c.E > 0
    K = c.K
    for k in [0, 1, 31, 32, 95] + [int(p) % K for p in c.esc_pos[:5]]:
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80  # 1.0
        y = O.gemv_container(c, x)
        col = np.array([_f(v) for v in w[:, k]])
        assert np.array_equal(y[0], col)
    y0 = O.gemv_container(c, np.zeros((4, K), np.uint16))
    assert not y0.any()
    # linearity: y(2x) = 2 y(x) exactly (scaling by 2 is exact)
    x = synth.gen_x_np(2, K, 3)
    x2 = synth.f32_to_bf16_bits(2 * synth.bf16_bits_to_f32(x))
    assert np.array_equal(O.gemv_container(c, x2), 2 * O.gemv_container(c, x))


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_decode_rows_matches_full(scheme):
    w = synth.gen_weights_np(synth.WeightSpec("t", 12, 1000, "t4", 0.02, 0.01, "normal", 1.0, seed=4))
    c = O.encode(w, scheme)
    rows = np.array([0, 3, 11])
    assert np.array_equal(O.decode_rows(c, rows), w[rows])


def test_synth_rounding_matches_ieee_rne():
    # ties to even at the BF16 boundary, values read with struct (not numpy views)
    cases = {0x3F808000: 0x3F80, 0x3F818000: 0x3F82, 0x3F808001: 0x3F81, 0x3F80FFFF: 0x3F81,
             0x7F7FFFFF: 0x7F80, 0xBF808000: 0xBF80}
    for u, b in cases.items():
        f = struct.unpack("<f", struct.pack("<I", u))[0]
        assert int(synth.f32_to_bf16_bits(np.array([f], np.float32))[0]) == b


def test_dense12_workload_has_no_byte_split_escape():
    """The escape-free workload of the dense 12-bit ablation: every magnitude in
    [2^-14, 2^-2) leaves 14 high bytes (two signs x exponent bits 7..1 of
    113..124), fewer than the table's 15, so byte-split escapes nothing and
    costs 4 + 8 + 15 * 8 / n bits per weight."""
    w = synth.gen_weights_np(synth.dense12_spec(64, 2048, seed=3))
    hi = np.unique(w >> 8)
    assert len(hi) <= 14
    c = O.encode(w, O.BYTESPLIT)
    assert c.E == 0
    assert O.entropy_bpw(O.BYTESPLIT, c.n, c.E) == pytest.approx(12 + 15 * 8 / c.n)
    assert np.array_equal(O.decode(c).reshape(w.shape), w)
