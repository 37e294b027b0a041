"""CPU oracle for lossless BF16 weight coding (byte-split and K15) and its GEMV.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the CUDA library computes.  Only the test suite, the smoke
check and the benchmark's CPU-baseline leg may import it; the library never
does, and the two share no code.  It is written with numpy array operations
(one library primitive per step: bincount, lexsort, matmul) and keeps every
step in the order the method states it.

The method (sources, cited by page title and section):

* "Prueba de GLM-5.2 reduce la memoria BF16 en casi un 25%" (forgeeks.dev),
  section "Cómo funciona la compresión":
  - a BF16 weight is 1 sign bit, 8 exponent bits and 7 mantissa bits, and
    trained weights reuse a small set of sign+exponent combinations;
  - K15: the 9-bit sign+exponent symbol becomes a 4-bit code that points
    into a 15-entry table; rare 9-bit symbols go to an exact escape stream;
    the 7-bit mantissa is stored uncompressed (11.173 bits/weight with all
    overhead on the pages' checkpoint);
  - byte-split: the high byte is rebuilt from a dictionary of codes,
    indices and an escape stream, and the low byte is left unchanged
    (12.005 bits/weight, 24.967% below BF16, every tensor bit-exact).
* "Compresión de pesos LLM sin pérdida vs 8-bit GGUF" (wavect.io), section
  "¿Qué significa “sin pérdida” para los pesos de un LLM?": lossless means
  the round trip rebuilds every bit of the BF16 tensor; the GPU may keep the
  weights encoded and rebuild exact BF16 in registers for the matmul.

Readings where the pages are silent (each is listed in the design notes):

* one table per tensor; the table is the 15 most frequent symbols ordered
  by (count descending, symbol ascending), with never-seen symbols filling
  it in ascending order when fewer than 15 occur; code 15 is the escape;
* the escape stream holds (position, value) pairs in ascending position;
  for byte-split the value is the high byte, for K15 the value is the whole
  16-bit word (its top 9 bits are the symbol, the low 7 repeat the raw
  mantissa so the weight can be rebuilt from the entry alone);
* the physical container layout (nibble order, K15 mantissa bytes, indexes,
  header, checksums) is this library's own and is defined here; it has two
  serialized forms: version 1 keeps the (position, value) escape stream and
  both indexes, version 2 (compact) keeps only what the pages count: the
  escape symbols at their symbol width (8 bits, or 9 bits packed for K15)
  and one 16-bit escape count per tile, with every position implied by its
  code 15 (forgeeks page, "Cómo funciona la compresión": the escape stream
  holds the rare symbols exactly; its bits/weight counts them at symbol
  width);
* the GEMV is y[b, r] = sum_k x[b, k] * W[r, k] evaluated in float64 from
  the exact BF16 values (accumulation order is not part of the method).

Parity is pinned (not by re-typing these formulas) in tests/test_oracle_*.py:
brute force over all 65,536 BF16 patterns, per-element pure-Python readers of
the serialized bytes, closed forms of the stream sizes, the pages' bit
accounting identities and one-hot / zero GEMV cases.
"""
from __future__ import annotations

import dataclasses
import struct
import zlib
from typing import Optional, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# Format constants of container version 1.
# ---------------------------------------------------------------------------
MAGIC = b"WCMP"
VERSION = 1
VERSION_COMPACT = 2
BYTESPLIT = 0
K15 = 1
SCHEMES = (BYTESPLIT, K15)
TABLE_SIZE = 15
ESCAPE = 15
TILE = 8192  # elements per decode tile (granule of the tile escape index)
GROUP = 32  # elements per K15 mantissa group (28 bytes)
HEADER_BYTES = 96
ALIGN = 32  # every payload section starts on a 32-byte boundary (256-bit loads)

SYM_BITS = {BYTESPLIT: 8, K15: 9}
RAW_BITS = {BYTESPLIT: 8, K15: 7}
NBINS = {BYTESPLIT: 256, K15: 512}


def _pad(nbytes: int) -> int:
    return (nbytes + ALIGN - 1) // ALIGN * ALIGN


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


# ---------------------------------------------------------------------------
# Step 1 - split each BF16 word into the coded symbol and the raw bits.
# ---------------------------------------------------------------------------
def split_symbols(w: np.ndarray, scheme: int) -> Tuple[np.ndarray, np.ndarray]:
    """Symbol and raw bits of every weight.

    byte-split: symbol = high byte (sign + exponent bits 7..1), raw = low byte.
    K15: symbol = 9-bit sign+exponent, raw = 7-bit mantissa.
    """
    w = np.asarray(w, dtype=np.uint16).reshape(-1).astype(np.uint32)
    if scheme == BYTESPLIT:
        return w >> 8, w & 0xFF
    if scheme == K15:
        return w >> 7, w & 0x7F
    raise ValueError(f"unknown scheme {scheme}")


# ---------------------------------------------------------------------------
# Step 2 - histogram of symbols over the tensor.
# ---------------------------------------------------------------------------
def histogram(sym: np.ndarray, scheme: int) -> np.ndarray:
    """Count of every possible symbol (256 high bytes / 512 sign+exponent values).

    forgeeks page, "Cómo funciona la compresión": the table holds the most reused sign+exponent
    combinations, which is a count over the tensor (one table per tensor is
    the reading taken where the page does not say)."""
    return np.bincount(sym, minlength=NBINS[scheme]).astype(np.int64)


# ---------------------------------------------------------------------------
# Step 3 - the 15-entry table: most frequent symbols first.
# ---------------------------------------------------------------------------
def select_table(hist: np.ndarray) -> np.ndarray:
    """Order all bins by (count descending, symbol ascending); keep the first 15.

    forgeeks page, "Cómo funciona la compresión": 15 table entries addressed by a
    4-bit code.  The tie-break and the filling with unseen symbols are the
    readings taken where the page is silent."""
    syms = np.arange(hist.size)
    order = np.lexsort((syms, -hist))  # last key is primary
    return order[:TABLE_SIZE].astype(np.uint32)


# ---------------------------------------------------------------------------
# Step 4 - codes: table index of each symbol, 15 (escape) when absent.
# ---------------------------------------------------------------------------
def assign_codes(sym: np.ndarray, table: np.ndarray, scheme: int) -> np.ndarray:
    """Code of every element: its table index, or 15 (escape) for a symbol
    outside the table.  forgeeks page, "Cómo funciona la compresión": a 4-bit code
    into a 15-entry table, rare symbols to an exact escape stream (code 15 as
    the escape marker is the reading of a 4-bit code that addresses 15 entries)."""
    lut = np.full(NBINS[scheme], ESCAPE, dtype=np.uint8)
    lut[table] = np.arange(TABLE_SIZE, dtype=np.uint8)
    return lut[sym]


# ---------------------------------------------------------------------------
# Step 5 - streams.
# ---------------------------------------------------------------------------
def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte: element 2j in the low nibble, 2j+1 in the high nibble.

    The 4-bit code stream of the forgeeks page ("Cómo funciona la compresión");
    the nibble order is this library's layout."""
    c = codes.astype(np.uint8)
    if c.size % 2:
        c = np.concatenate([c, np.zeros(1, np.uint8)])
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8)


def pack_k15_planes(raw7: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The 7 mantissa bits of every element, 28 bytes per 32-element group.

    The pages store the K15 mantissa uncompressed at 7 bits per weight but
    give it no physical layout; this is the library's own.  Elements are taken
    in groups of 32 (the last group zero padded).  Byte j (j < 28) of a group
    holds element j's mantissa in bits 0..6; bit 7 of byte j holds bit
    j // 4 of the mantissa of element 28 + j % 4.  So element 28 + i is spread
    over bit 7 of bytes i, 4 + i, ..., 24 + i (its bits 0 .. 6), and byte j
    sits in byte lane j % 4 of 32-bit word j // 4.

    The 28 bytes are split into three sections with power-of-two strides:
    ``plane_a`` bytes 0..15 (16 per group), ``plane_b`` bytes 16..23 (8 per
    group) and ``plane_c`` bytes 24..27 (4 per group).
    """
    n = raw7.size
    groups = _cdiv(n, GROUP)
    m = np.zeros(groups * GROUP, dtype=np.uint32)
    m[:n] = raw7
    m = m.reshape(groups, GROUP)
    j = np.arange(28)
    tail_bit = (m[:, 28 + (j % 4)] >> (j // 4)) & 1  # [group, byte j]
    mb = (m[:, :28] | (tail_bit << 7)).astype(np.uint8)
    return (mb[:, :16].reshape(-1).copy(), mb[:, 16:24].reshape(-1).copy(), mb[:, 24:28].reshape(-1).copy())


def unpack_k15_planes(pa: np.ndarray, pb: np.ndarray, pc: np.ndarray, n: int) -> np.ndarray:
    """Inverse of :func:`pack_k15_planes` (returns the n 7-bit mantissas)."""
    groups = _cdiv(n, GROUP)
    mb = np.concatenate([np.asarray(pa[: 16 * groups], np.uint8).reshape(groups, 16),
                         np.asarray(pb[: 8 * groups], np.uint8).reshape(groups, 8),
                         np.asarray(pc[: 4 * groups], np.uint8).reshape(groups, 4)], axis=1).astype(np.uint32)
    head = mb & 0x7F  # elements 0..27
    tail = np.zeros((groups, 4), dtype=np.uint32)  # elements 28..31
    for b in range(7):
        tail |= ((mb[:, 4 * b:4 * b + 4] >> 7) & 1) << b
    m = np.concatenate([head, tail], axis=1).reshape(-1)
    return m[:n].astype(np.uint32)


def escape_index(pos: np.ndarray, bounds: np.ndarray) -> np.ndarray:
    """entry j = number of escapes whose position is below bounds[j].

    Not part of the method's definition: an index over the escape stream so a
    decoder finds a tile's or a row's escapes without a search (layout of
    this library; the escape stream itself is the forgeeks page's, "Cómo
    funciona la compresión")."""
    return np.searchsorted(pos, bounds, side="left").astype(np.uint32)


# ---------------------------------------------------------------------------
# The container.
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Container:
    scheme: int
    N: int
    K: int
    table: np.ndarray  # uint32[15]
    codes: np.ndarray  # uint8[ceil(n/2)]
    raw: np.ndarray  # byte-split: uint8[n]
    plane_a: Optional[np.ndarray]  # K15 planes
    plane_b: Optional[np.ndarray]
    plane_c: Optional[np.ndarray]
    tile_index: np.ndarray  # uint32[n_tiles + 1]
    row_index: np.ndarray  # uint32[N + 1]
    esc_pos: np.ndarray  # uint32[E]
    esc_val: np.ndarray  # uint8[E] (byte-split) / uint16[E] (K15)
    hist: np.ndarray  # int64[nbins] (diagnostic, not serialized)

    @property
    def n(self) -> int:
        return self.N * self.K

    @property
    def E(self) -> int:
        return int(self.esc_pos.size)

    @property
    def n_tiles(self) -> int:
        return _cdiv(self.n, TILE)


def encode(w: np.ndarray, scheme: int, N: Optional[int] = None, K: Optional[int] = None) -> Container:
    """Encode BF16 bits w (any shape; read as W[N, K], default N=1 row if 1-D).

    The steps of forgeeks page, "Cómo funciona la compresión", in its order: split
    each weight into the coded symbol and the raw bits, count the symbols, keep
    the 15 most frequent as the table, code every element (15 = escape), and
    keep the escaped symbols exactly in their own stream."""
    w = np.asarray(w, dtype=np.uint16)
    if N is None or K is None:
        if w.ndim == 2:
            N, K = w.shape
        else:
            N, K = 1, w.size
    n = N * K
    if n != w.size:
        raise ValueError("shape does not match element count")
    if not 0 < n < 2**32:
        raise ValueError("element count must be in [1, 2^32)")
    sym, raw = split_symbols(w, scheme)
    hist = histogram(sym, scheme)
    table = select_table(hist)
    codes = assign_codes(sym, table, scheme)
    packed = pack_nibbles(codes)
    esc_pos = np.flatnonzero(codes == ESCAPE).astype(np.uint32)
    wf = w.reshape(-1)
    if scheme == BYTESPLIT:
        raw_bytes = raw.astype(np.uint8)
        pa = pb = pc = None
        esc_val = sym[esc_pos].astype(np.uint8)
    else:
        raw_bytes = np.zeros(0, np.uint8)
        pa, pb, pc = pack_k15_planes(raw)
        esc_val = wf[esc_pos].astype(np.uint16)
    n_tiles = _cdiv(n, TILE)
    tile_index = escape_index(esc_pos, np.arange(n_tiles + 1, dtype=np.int64) * TILE)
    row_index = escape_index(esc_pos, np.arange(N + 1, dtype=np.int64) * K)
    return Container(scheme, N, K, table, packed, raw_bytes, pa, pb, pc,
                     tile_index, row_index, esc_pos, esc_val, hist)


# ---------------------------------------------------------------------------
# Decode.
# ---------------------------------------------------------------------------
def unpack_codes(packed: np.ndarray, n: int) -> np.ndarray:
    """Inverse of :func:`pack_nibbles`."""
    c = np.empty(2 * packed.size, dtype=np.uint8)
    c[0::2] = packed & 0xF
    c[1::2] = packed >> 4
    return c[:n]


def decode(c: Container) -> np.ndarray:
    """Rebuild the exact BF16 bits, shape [N, K].

    Table symbol (or the escape stream's symbol) above the raw bits: the
    forgeeks page, "Cómo funciona la compresión"; lossless means every bit
    comes back (wavect page, "¿Qué significa “sin pérdida” para los pesos de
    un LLM?")."""
    n = c.n
    codes = unpack_codes(c.codes, n)
    table = c.table.astype(np.uint32)
    sym = np.where(codes < ESCAPE, table[np.minimum(codes, TABLE_SIZE - 1)], 0).astype(np.uint32)
    if c.scheme == BYTESPLIT:
        sym[c.esc_pos] = c.esc_val.astype(np.uint32)
        w = (sym << 8) | c.raw[:n].astype(np.uint32)
    else:
        raw = unpack_k15_planes(c.plane_a, c.plane_b, c.plane_c, n)
        w = (sym << 7) | raw
        w[c.esc_pos] = c.esc_val.astype(np.uint32)
    return w.astype(np.uint16).reshape(c.N, c.K)


def decode_rows(c: Container, rows: np.ndarray) -> np.ndarray:
    """Exact BF16 bits of the selected rows only (for sampled checks at full size)."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, c.K), dtype=np.uint16)
    table = c.table.astype(np.uint32)
    for j, r in enumerate(rows):
        a, b = int(r) * c.K, (int(r) + 1) * c.K
        idx = np.arange(a, b, dtype=np.int64)
        nib = c.codes[idx >> 1]
        code = np.where(idx & 1, nib >> 4, nib & 0xF).astype(np.uint8)
        sym = np.where(code < ESCAPE, table[np.minimum(code, TABLE_SIZE - 1)], 0).astype(np.uint32)
        e0, e1 = int(c.row_index[r]), int(c.row_index[r + 1])
        epos = c.esc_pos[e0:e1].astype(np.int64) - a
        if c.scheme == BYTESPLIT:
            sym[epos] = c.esc_val[e0:e1].astype(np.uint32)
            w = (sym << 8) | c.raw[a:b].astype(np.uint32)
        else:
            g0, g1 = a // GROUP, _cdiv(b, GROUP)
            raw = unpack_k15_planes(c.plane_a[16 * g0:16 * g1], c.plane_b[8 * g0:8 * g1],
                                    c.plane_c[4 * g0:4 * g1], (g1 - g0) * GROUP)
            raw = raw[a - g0 * GROUP: b - g0 * GROUP]
            w = (sym << 7) | raw
            w[epos] = c.esc_val[e0:e1].astype(np.uint32)
        out[j] = w.astype(np.uint16)
    return out


# ---------------------------------------------------------------------------
# Serialization (container version 1).
# ---------------------------------------------------------------------------
def section_sizes(scheme: int, N: int, K: int, E: int) -> list:
    """Unpadded byte size of every payload section, in payload order."""
    n = N * K
    groups = _cdiv(n, GROUP)
    if scheme == BYTESPLIT:
        raw = [("raw", n)]
        val = E
    else:
        raw = [("plane_a", 16 * groups), ("plane_b", 8 * groups), ("plane_c", 4 * groups)]
        val = 2 * E
    return ([("codes", _cdiv(n, 2))] + raw +
            [("tile_index", 4 * (_cdiv(n, TILE) + 1)), ("row_index", 4 * (N + 1)),
             ("esc_pos", 4 * E), ("esc_val", val)])


def serialize(c: Container) -> bytes:
    """Container version 1: header, then codes, raw bytes or K15 planes, both
    indexes, escape positions and values, each section padded to 32 bytes.
    The pages define no file format; this layout is the library's own."""
    parts = [("codes", c.codes)]
    if c.scheme == BYTESPLIT:
        parts.append(("raw", c.raw))
    else:
        parts += [("plane_a", c.plane_a), ("plane_b", c.plane_b), ("plane_c", c.plane_c)]
    parts += [("tile_index", c.tile_index.astype("<u4").view(np.uint8)),
              ("row_index", c.row_index.astype("<u4").view(np.uint8)),
              ("esc_pos", c.esc_pos.astype("<u4").view(np.uint8)),
              ("esc_val", (c.esc_val.astype(np.uint8) if c.scheme == BYTESPLIT
                           else c.esc_val.astype("<u2").view(np.uint8)))]
    sizes = section_sizes(c.scheme, c.N, c.K, c.E)
    payload = bytearray()
    for (name, arr), (name2, size) in zip(parts, sizes):
        assert name == name2 and arr.size == size, (name, arr.size, size)
        payload += arr.tobytes()
        payload += b"\0" * (_pad(size) - size)
    return _header(VERSION, c, bytes(payload)) + bytes(payload)


class CorruptContainer(ValueError):
    pass


def deserialize(buf: bytes) -> Container:
    """Parse and fully validate either serialized form (checksums, sizes, the
    table, ascending in-range positions, indexes and codes agreeing with the
    escape stream); raise CorruptContainer on any mismatch.  The wavect page
    ("Un piloto de producción de 14 días") asks for corruption to be caught
    before use."""
    if len(buf) < HEADER_BYTES:
        raise CorruptContainer("short header")
    head = buf[:HEADER_BYTES]
    if head[:4] != MAGIC:
        raise CorruptContainer("bad magic")
    if struct.unpack_from("<I", head, 92)[0] != zlib.crc32(head[:92]):
        raise CorruptContainer("header checksum")
    version, scheme, _ = struct.unpack_from("<HBB", head, 4)
    if version not in (VERSION, VERSION_COMPACT) or scheme not in SCHEMES:
        raise CorruptContainer("version/scheme")
    N, K, E = struct.unpack_from("<qqQ", head, 8)
    tile, _ = struct.unpack_from("<II", head, 32)
    table = np.array(struct.unpack_from("<15H", head, 40), dtype=np.uint32)
    plen, pcrc = struct.unpack_from("<QI", head, 72)
    if tile != TILE or N <= 0 or K <= 0 or not N * K < 2**32 or E > N * K:
        raise CorruptContainer("sizes")
    if len(set(table.tolist())) != TABLE_SIZE or int(table.max()) >= NBINS[scheme]:
        raise CorruptContainer("table")
    if version == VERSION_COMPACT:
        return _deserialize_compact(buf, scheme, N, K, E, table, plen, pcrc)
    sizes = section_sizes(scheme, N, K, E)
    if plen != sum(_pad(s) for _, s in sizes) or len(buf) != HEADER_BYTES + plen:
        raise CorruptContainer("payload length")
    payload = np.frombuffer(buf, dtype=np.uint8, offset=HEADER_BYTES)
    if zlib.crc32(payload.tobytes()) != pcrc:
        raise CorruptContainer("payload checksum")
    sec = {}
    off = 0
    for name, size in sizes:
        sec[name] = payload[off: off + size]
        off += _pad(size)
    n = N * K
    esc_pos = sec["esc_pos"].view("<u4").astype(np.uint32)
    esc_val = sec["esc_val"].copy() if scheme == BYTESPLIT else sec["esc_val"].view("<u2").astype(np.uint16)
    tile_index = sec["tile_index"].view("<u4").astype(np.uint32)
    row_index = sec["row_index"].view("<u4").astype(np.uint32)
    if E and (np.any(np.diff(esc_pos.astype(np.int64)) <= 0) or int(esc_pos[-1]) >= n):
        raise CorruptContainer("escape positions")
    n_tiles = _cdiv(n, TILE)
    if not np.array_equal(tile_index, escape_index(esc_pos, np.arange(n_tiles + 1, dtype=np.int64) * TILE)):
        raise CorruptContainer("tile index")
    if not np.array_equal(row_index, escape_index(esc_pos, np.arange(N + 1, dtype=np.int64) * K)):
        raise CorruptContainer("row index")
    if len(set(table.tolist())) != TABLE_SIZE or int(table.max()) >= NBINS[scheme]:
        raise CorruptContainer("table")
    codes = sec["codes"].copy()
    if not np.array_equal(np.flatnonzero(unpack_codes(codes, n) == ESCAPE).astype(np.uint32), esc_pos):
        raise CorruptContainer("escape codes")
    if scheme == BYTESPLIT:
        return Container(scheme, N, K, table, codes, sec["raw"].copy(), None, None, None,
                         tile_index, row_index, esc_pos, esc_val, np.zeros(0, np.int64))
    return Container(scheme, N, K, table, codes, np.zeros(0, np.uint8),
                     sec["plane_a"].copy(), sec["plane_b"].copy(), sec["plane_c"].copy(),
                     tile_index, row_index, esc_pos, esc_val, np.zeros(0, np.int64))


# ---------------------------------------------------------------------------
# Compact serialized form (version 2): no positions, no row index.
# ---------------------------------------------------------------------------
def pack_bits9(vals: np.ndarray) -> np.ndarray:
    """9-bit values into a little-endian bit stream: value r occupies stream
    bits 9r .. 9r+8, least significant first; stream bit b is bit (b % 8) of
    byte b // 8.  The last byte is zero-padded."""
    vals = np.asarray(vals, dtype=np.uint32)
    bits = ((vals[:, None] >> np.arange(9, dtype=np.uint32)) & 1).astype(np.uint8).reshape(-1)
    out = np.zeros(_cdiv(bits.size, 8), dtype=np.uint8)
    if bits.size:
        padded = np.zeros(out.size * 8, dtype=np.uint8)
        padded[: bits.size] = bits
        out = np.packbits(padded.reshape(-1, 8), axis=1, bitorder="little").reshape(-1)
    return out


def unpack_bits9(buf: np.ndarray, count: int) -> np.ndarray:
    """Inverse of :func:`pack_bits9`: the first ``count`` 9-bit values."""
    bits = np.unpackbits(np.asarray(buf, dtype=np.uint8), bitorder="little")[: 9 * count]
    return (bits.reshape(count, 9).astype(np.uint32) << np.arange(9, dtype=np.uint32)).sum(axis=1).astype(np.uint32)


def section_sizes_compact(scheme: int, N: int, K: int, E: int) -> list:
    """Unpadded byte size of every payload section of the compact form, in order."""
    n = N * K
    groups = _cdiv(n, GROUP)
    if scheme == BYTESPLIT:
        raw = [("raw", n)]
        sym = E
    else:
        raw = [("plane_a", 16 * groups), ("plane_b", 8 * groups), ("plane_c", 4 * groups)]
        sym = _cdiv(9 * E, 8)
    return [("codes", _cdiv(n, 2))] + raw + [("tile_count", 2 * _cdiv(n, TILE)), ("esc_sym", sym)]


def _header(version: int, c: "Container", payload: bytes) -> bytes:
    table16 = struct.pack("<15H", *[int(t) for t in c.table])
    head = (MAGIC + struct.pack("<HBB", version, c.scheme, 0) +
            struct.pack("<qqQ", c.N, c.K, c.E) + struct.pack("<II", TILE, 0) +
            table16 + struct.pack("<H", 0) +
            struct.pack("<QI", len(payload), zlib.crc32(payload)) + b"\0" * 8)
    assert len(head) == 92
    return head + struct.pack("<I", zlib.crc32(head))


def serialize_compact(c: Container) -> bytes:
    """Version 2: codes, raw bytes or K15 planes, the escape count of every
    tile (u16; a tile holds at most 8192 escapes) and the escape symbols in
    ascending position order (byte-split: the high byte; K15: the 9-bit
    symbol, the top 9 bits of the escaped word, packed by pack_bits9)."""
    parts = [("codes", c.codes)]
    if c.scheme == BYTESPLIT:
        parts.append(("raw", c.raw))
        sym = c.esc_val.astype(np.uint8)
    else:
        parts += [("plane_a", c.plane_a), ("plane_b", c.plane_b), ("plane_c", c.plane_c)]
        sym = pack_bits9(c.esc_val.astype(np.uint32) >> 7)
    parts += [("tile_count", np.diff(c.tile_index.astype(np.int64)).astype("<u2").view(np.uint8)),
              ("esc_sym", sym)]
    payload = bytearray()
    for (name, arr), (name2, size) in zip(parts, section_sizes_compact(c.scheme, c.N, c.K, c.E)):
        assert name == name2 and arr.size == size, (name, arr.size, size)
        payload += arr.tobytes()
        payload += b"\0" * (_pad(size) - size)
    return _header(VERSION_COMPACT, c, bytes(payload)) + bytes(payload)


def _deserialize_compact(buf: bytes, scheme: int, N: int, K: int, E: int, table: np.ndarray,
                         plen: int, pcrc: int) -> Container:
    sizes = section_sizes_compact(scheme, N, K, E)
    if plen != sum(_pad(s) for _, s in sizes) or len(buf) != HEADER_BYTES + plen:
        raise CorruptContainer("payload length")
    payload = np.frombuffer(buf, dtype=np.uint8, offset=HEADER_BYTES)
    if zlib.crc32(payload.tobytes()) != pcrc:
        raise CorruptContainer("payload checksum")
    sec = {}
    off = 0
    for name, size in sizes:
        sec[name] = payload[off: off + size]
        off += _pad(size)
    n = N * K
    codes = sec["codes"].copy()
    # every position is implied by its code 15
    esc_pos = np.flatnonzero(unpack_codes(codes, n) == ESCAPE).astype(np.uint32)
    if esc_pos.size != E:
        raise CorruptContainer("escape count")
    n_tiles = _cdiv(n, TILE)
    tile_index = escape_index(esc_pos, np.arange(n_tiles + 1, dtype=np.int64) * TILE)
    counts = sec["tile_count"].view("<u2").astype(np.int64)
    if not np.array_equal(counts, np.diff(tile_index.astype(np.int64))):
        raise CorruptContainer("tile counts")
    row_index = escape_index(esc_pos, np.arange(N + 1, dtype=np.int64) * K)
    if scheme == BYTESPLIT:
        esc_val = sec["esc_sym"].copy()
        return Container(scheme, N, K, table, codes, sec["raw"].copy(), None, None, None,
                         tile_index, row_index, esc_pos, esc_val, np.zeros(0, np.int64))
    sym9 = unpack_bits9(sec["esc_sym"], E)
    pa, pb, pc = sec["plane_a"].copy(), sec["plane_b"].copy(), sec["plane_c"].copy()
    mant = unpack_k15_planes(pa, pb, pc, n)[esc_pos] if E else np.zeros(0, np.uint32)
    esc_val = ((sym9 << 7) | mant).astype(np.uint16)
    return Container(scheme, N, K, table, codes, np.zeros(0, np.uint8), pa, pb, pc,
                     tile_index, row_index, esc_pos, esc_val, np.zeros(0, np.int64))


def serialized_len_compact(scheme: int, N: int, K: int, E: int) -> int:
    """Byte length of the compact form for these sizes."""
    return HEADER_BYTES + sum(_pad(s) for _, s in section_sizes_compact(scheme, N, K, E))


# ---------------------------------------------------------------------------
# GEMV in float64 from the exact BF16 values.
# ---------------------------------------------------------------------------
def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact value of BF16 bits (BF16 is the top half of an fp32 word)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemv(w_bits: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """y[B, N] = x[B, K] @ W[N, K].T in float64.

    The product the fused kernel computes with W rebuilt from the codes
    (forgeeks page, "Qué queda por demostrar"), stated on the exact BF16
    values; every product of two BF16 numbers and every partial sum here is
    far more precise than the fp32 arithmetic it is compared with."""
    W = bf16_to_f64(w_bits)
    X = bf16_to_f64(x_bits)
    return X @ W.T


def gemv_container(c: Container, x_bits: np.ndarray, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """GEMV through the container: decode (all rows, or the selected rows), then float64 matmul."""
    if rows is None:
        return gemv(decode(c), x_bits)
    return gemv(decode_rows(c, rows), x_bits)


# ---------------------------------------------------------------------------
# Bit accounting.
# ---------------------------------------------------------------------------
def entropy_bpw(scheme: int, n: int, E: int) -> float:
    """Bits per weight as the pages count them: 4 code bits + raw bits, plus the
    table (15 symbols) and every escape at its symbol width (the escape position
    is implied by code 15)."""
    return 4 + RAW_BITS[scheme] + (E * SYM_BITS[scheme] + TABLE_SIZE * SYM_BITS[scheme]) / n


def physical_bpw(serialized_len: int, n: int) -> float:
    """Bits per weight of a serialized container, every byte counted."""
    return 8.0 * serialized_len / n


def serialized_len(scheme: int, N: int, K: int, E: int) -> int:
    """Byte length of container version 1 for these sizes."""
    return HEADER_BYTES + sum(_pad(s) for _, s in section_sizes(scheme, N, K, E))


def reduction_pct(bpw: float) -> float:
    """Size reduction against 16-bit BF16, in percent."""
    return 100.0 * (1.0 - bpw / 16.0)
