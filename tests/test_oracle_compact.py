"""Pins for the compact serialized form (version 2) of the oracle.

The compact form keeps what the pages' bit accounting counts: the escape
symbols at their symbol width, with every position implied by its code 15
(forgeeks page "Prueba de GLM-5.2 reduce la memoria BF16 en casi un 25%",
section "Cómo funciona la compresión").  Pinned here by a hand-derived bit
packing example, closed-form sizes, an independent pure-Python reader that
walks the bytes element by element (escape symbols consumed in order, and
each tile's stored count checked against the escapes met in that tile), the
bits/weight bound against the entropy accounting, and corruption cases.
"""
import struct
import zlib

import numpy as np
import pytest

from decode_gemv_sign_gb300 import synth
from oracle import wcomp_oracle as O


def _pad(x):
    return (x + 31) // 32 * 32


def read_all_compact_pure(buf: bytes) -> list:
    """Every weight of a compact container, rebuilt with plain integer code:
    the r-th code 15 met in element order takes the r-th escape symbol."""
    assert struct.unpack_from("<H", buf, 4)[0] == 2
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
    tc_off = p
    n_tiles = (n + 8191) // 8192
    p += _pad(2 * n_tiles)
    sym_off = p
    out = []
    r = 0
    per_tile = [0] * n_tiles
    for i in range(n):
        byte = buf[codes_off + i // 2]
        code = (byte >> 4) if i % 2 else (byte & 15)
        per_tile[i // 8192] += code == 15
        if scheme == 0:
            low = buf[raw_off + i]
        else:
            g, e = divmod(i, 32)
            def mbyte(j):
                if j < 16:
                    return buf[a_off + 16 * g + j]
                if j < 24:
                    return buf[b_off + 8 * g + j - 16]
                return buf[c_off + 4 * g + j - 24]
            low = (mbyte(e) & 0x7F) if e < 28 else sum(((mbyte(4 * b + e - 28) >> 7) & 1) << b for b in range(7))
        if code != 15:
            sym = table[code]
        elif scheme == 0:
            sym = buf[sym_off + r]
            r += 1
        else:
            bit = 9 * r
            word = int.from_bytes(buf[sym_off + bit // 8: sym_off + bit // 8 + 2], "little")
            sym = (word >> (bit % 8)) & 0x1FF
            r += 1
        out.append((sym << 8) | low if scheme == 0 else (sym << 7) | low)
    assert r == E
    # the count section holds each 8192-element tile's own number of escapes
    assert list(struct.unpack_from(f"<{n_tiles}H", buf, tc_off)) == per_tile
    return out


def test_pack_bits9_hand_example():
    # 0x1FF, 0x000, 0x155, 0x0AA at stream bits 0-8, 9-17, 18-26, 27-35:
    # byte 0 = bits 0-7 all set; byte 1 = bit 8 set; byte 2 = bits 18, 20, 22;
    # byte 3 = bits 24, 26, 28, 30; byte 4 = bits 32, 34.
    got = O.pack_bits9(np.array([0x1FF, 0x000, 0x155, 0x0AA]))
    assert got.tolist() == [0xFF, 0x01, 0x54, 0x55, 0x05]
    assert O.unpack_bits9(got, 4).tolist() == [0x1FF, 0x000, 0x155, 0x0AA]
    # the values above read the same in either bit order; these do not:
    # 0x001 sets stream bit 0; 0x100 sets bit 9 + 8 = 17; 0x003 sets bits 18 and 19
    # -> byte 0 = 0x01, byte 2 = bits 1, 2, 3 = 0x0E, 27 bits in 4 bytes
    got = O.pack_bits9(np.array([0x001, 0x100, 0x003]))
    assert got.tolist() == [0x01, 0x00, 0x0E, 0x00]
    assert O.unpack_bits9(got, 3).tolist() == [0x001, 0x100, 0x003]
    vals = np.random.default_rng(3).integers(0, 512, 1001)
    assert np.array_equal(O.unpack_bits9(O.pack_bits9(vals), vals.size), vals)
    assert O.pack_bits9(np.zeros(0)).size == 0


def test_compact_size_closed_form():
    # N=2, K=16: codes 16 B, tile counts 2 B, each section padded to 32 B.
    w = np.zeros(32, np.uint16)
    c = O.encode(w, O.BYTESPLIT, 2, 16)
    assert c.E == 0 and len(O.serialize_compact(c)) == 96 + 32 + 32 + 32 + 0
    # K15 with 3 escapes: planes 16 + 8 + 4 B, symbols ceil(27 / 8) = 4 B.
    w = np.zeros(32, np.uint16)
    w[:15] = np.arange(15) << 7
    w[[20, 25, 31]] = [0x5000, 0x5080, 0x5100]
    c = O.encode(w, O.K15, 2, 16)
    assert c.E == 3
    assert len(O.serialize_compact(c)) == 96 + 32 + 3 * 32 + 32 + 32
    assert O.serialized_len_compact(O.K15, 2, 16, 3) == 288


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_compact_pure_reader_all_patterns(scheme):
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for arr in (w, np.random.default_rng(11).permutation(w)):
        c = O.encode(arr, scheme, 256, 256)
        buf = O.serialize_compact(c)
        assert read_all_compact_pure(buf) == arr.tolist()
        back = O.deserialize(buf)
        assert O.serialize(back) == O.serialize(c)


@pytest.mark.parametrize("scheme", O.SCHEMES)
@pytest.mark.parametrize("n", [1, 2, 3, 31, 33, 8191, 8193, 16385])
def test_compact_roundtrip_ragged(scheme, n):
    rng = np.random.default_rng(n)
    w = rng.integers(0, 65536, n).astype(np.uint16)
    w[: n // 2] = 0x3C00 | (w[: n // 2] & 0xFF)
    c = O.encode(w, scheme)
    back = O.deserialize(O.serialize_compact(c))
    assert O.serialize(back) == O.serialize(c)
    assert np.array_equal(O.decode(back).reshape(-1), w)


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_compact_bpw_against_entropy_accounting(scheme):
    spec = synth.WeightSpec("g", 1024, 1024, "normal", 0.02, 0.001, "normal", 0.5, 7)
    w = synth.gen_weights_np(spec)
    c = O.encode(w, scheme)
    n = c.n
    phys = O.physical_bpw(len(O.serialize_compact(c)), n)
    ent = O.entropy_bpw(scheme, n, c.E)
    # the compact form differs from the accounting only by the header, the
    # 32-byte section padding, the tile counts, the u16 table entries and the
    # byte rounding of the symbol stream
    sections = 3 if scheme == O.BYTESPLIT else 5
    bound = 8 * (96 + 31 * (sections + 1) + 2 * c.n_tiles + 1) / n
    assert ent - 8 * 30 / n <= phys <= ent + bound, (phys, ent)
    # and never above the version-1 form by less than its positions
    v1 = O.physical_bpw(len(O.serialize(c)), n)
    assert v1 - phys >= 8 * (4 * c.E + 4 * (c.N + 1)) / n - 8 * 64 / n


def _rewrite(buf: bytes, payload: bytes) -> bytes:
    head = bytearray(buf[:96])
    struct.pack_into("<I", head, 80, zlib.crc32(payload))
    struct.pack_into("<I", head, 92, zlib.crc32(bytes(head[:92])))
    return bytes(head) + payload


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_compact_corruption_detected(scheme):
    rng = np.random.default_rng(5)
    # 15 common symbols fill the table; three single rare symbols escape, in tiles 0, 1 and 2
    shift = 8 if scheme == O.BYTESPLIT else 7
    base = 0x30 if scheme == O.BYTESPLIT else 0x60
    w = ((rng.integers(base, base + 15, 3 * 8192) << shift) | rng.integers(0, 1 << shift, 3 * 8192)).astype(np.uint16)
    w[[10, 9000, 20000]] = [0x7F00, 0x7E80, 0x6100]
    c = O.encode(w, scheme)
    assert c.E >= 3
    buf = O.serialize_compact(c)
    # payload bit flip: checksum
    bad = bytearray(buf)
    bad[96 + 5] ^= 1
    with pytest.raises(O.CorruptContainer):
        O.deserialize(bytes(bad))
    payload = bytearray(buf[96:])
    # an escape code turned into code 0 (checksums recomputed): the count no longer matches E
    i = int(c.esc_pos[0])
    payload[i // 2] &= 0x0F if i % 2 else 0xF0
    with pytest.raises(O.CorruptContainer, match="escape count"):
        O.deserialize(_rewrite(buf, bytes(payload)))
    # an escape moved from tile 0 to tile 1 (E unchanged): the tile counts no longer match
    payload = bytearray(buf[96:])
    j = int(c.esc_pos[0])
    payload[j // 2] &= 0x0F if j % 2 else 0xF0
    k = 8192 + 1
    assert (O.unpack_codes(c.codes, c.n)[k]) != 15
    payload[k // 2] |= 0xF0 if k % 2 else 0x0F
    with pytest.raises(O.CorruptContainer, match="tile counts"):
        O.deserialize(_rewrite(buf, bytes(payload)))
