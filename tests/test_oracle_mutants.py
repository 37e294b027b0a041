"""The oracle's pins are strong enough: each plausible mistake, planted in the
oracle on the CPU, makes at least one independent pin fail.

A pin that passes whatever the oracle does proves nothing, so every mutant
below is a mistake a careful reader could still make (a reversed tie-break,
a swapped nibble or bit order that still round-trips, an index counted with
the wrong inequality, a dropped accounting term, fp32 instead of fp64
accumulation...).  Each is applied with monkeypatch to the oracle module only,
the pins of the two pin modules run against it, and the test asserts that one
of them fails.  The stored fixtures are left out on purpose: they were written
by the oracle itself and would catch any change without saying whether the
change was a mistake.
"""
import numpy as np
import pytest

import test_oracle_compact as PC
import test_oracle_pins as P
from oracle import wcomp_oracle as O

S = O.SCHEMES


def _pins():
    """(name, call) for every independent pin, cheap ones first."""
    out = [("k15_plane_bit_positions", P.test_k15_plane_bit_positions),
           ("nibble_order_fixture", P.test_nibble_order_fixture),
           ("pack_bits9_hand_example", PC.test_pack_bits9_hand_example),
           ("accounting_identities", P.test_accounting_identities_from_pages),
           ("gemv_brute_force_tiny", P.test_gemv_brute_force_tiny),
           ("gemv_exact_sum", P.test_gemv_is_exact_where_fp32_accumulation_is_not),
           ("synth_rounding", P.test_synth_rounding_matches_ieee_rne),
           ("compact_size_closed_form", PC.test_compact_size_closed_form),
           ("all_escape_except_table", P.test_all_escape_except_table)]
    for s in S:
        out += [(f"accounting_no_escapes[{s}]", lambda s=s: P.test_accounting_no_escapes_exact(s)),
                (f"special_values[{s}]", lambda s=s: P.test_special_values_roundtrip(s)),
                (f"histogram_table_brute_force[{s}]", lambda s=s: P.test_histogram_and_table_brute_force(s)),
                (f"escape_stream_and_indexes[{s}]", lambda s=s: P.test_escape_stream_and_indexes(s)),
                (f"indexes_on_boundaries[{s}]", lambda s=s: P.test_indexes_with_escapes_on_boundaries(s)),
                (f"decode_rows[{s}]", lambda s=s: P.test_decode_rows_matches_full(s)),
                (f"gemv_one_hot_and_zero[{s}]", lambda s=s: P.test_gemv_one_hot_and_zero(s)),
                (f"corruption[{s}]", lambda s=s: P.test_corruption_detected(s)),
                (f"compact_corruption[{s}]", lambda s=s: PC.test_compact_corruption_detected(s))]
        for d in (1, 15, 16, 17):
            out.append((f"distinct_symbols[{s},{d}]", lambda s=s, d=d: P.test_distinct_symbol_counts(s, d)))
        for n in (1, 2, 3, 31, 32, 33, 8191, 8192, 8193, 65537):
            out.append((f"ragged_roundtrip[{s},{n}]", lambda s=s, n=n: P.test_ragged_sizes_roundtrip(s, n)))
        for n in (1, 33, 8193):
            out.append((f"compact_ragged[{s},{n}]", lambda s=s, n=n: PC.test_compact_roundtrip_ragged(s, n)))
        out += [("accounting_gaussian", P.test_accounting_on_gaussian_weights_matches_pages),
                (f"serialized_size_closed_form[{s}]", lambda s=s: P.test_serialized_size_closed_form(s)),
                (f"compact_bpw_bound[{s}]", lambda s=s: PC.test_compact_bpw_against_entropy_accounting(s)),
                (f"all_65536_patterns[{s}]", lambda s=s: P.test_all_65536_patterns_roundtrip(s)),
                (f"compact_pure_reader[{s}]", lambda s=s: PC.test_compact_pure_reader_all_patterns(s))]
    return out


def _first_failing_pin():
    for name, call in _pins():
        try:
            call()
        except (Exception, pytest.fail.Exception):
            return name
    return None


# ---------------------------------------------------------------------------
# The planted mistakes.  Each returns {attribute of the oracle module: value}.
# ---------------------------------------------------------------------------
def _tie_break_descending():
    def select_table(hist):
        syms = np.arange(hist.size)
        return np.lexsort((-syms, -hist))[: O.TABLE_SIZE].astype(np.uint32)
    return {"select_table": select_table}


def _least_frequent_first():
    def select_table(hist):
        syms = np.arange(hist.size)
        return np.lexsort((syms, hist))[: O.TABLE_SIZE].astype(np.uint32)
    return {"select_table": select_table}


def _codes_off_by_one():
    def assign_codes(sym, table, scheme):
        lut = np.full(O.NBINS[scheme], O.ESCAPE, dtype=np.uint8)
        lut[table] = np.arange(1, O.TABLE_SIZE + 1, dtype=np.uint8)
        return lut[sym]
    return {"assign_codes": assign_codes}


def _histogram_without_empty_bins():
    return {"histogram": lambda sym, scheme: np.bincount(sym).astype(np.int64)}


def _k15_symbol_width_8():
    orig = O.split_symbols

    def split_symbols(w, scheme):
        if scheme == O.K15:
            w = np.asarray(w, dtype=np.uint16).reshape(-1).astype(np.uint32)
            return w >> 8, w & 0x7F
        return orig(w, scheme)
    return {"split_symbols": split_symbols}


def _nibbles_high_first():
    # consistent on both sides: still round-trips, but the byte layout is wrong
    def pack_nibbles(codes):
        c = codes.astype(np.uint8)
        if c.size % 2:
            c = np.concatenate([c, np.zeros(1, np.uint8)])
        return ((c[0::2] << 4) | c[1::2]).astype(np.uint8)

    def unpack_codes(packed, n):
        c = np.empty(2 * packed.size, dtype=np.uint8)
        c[0::2] = packed >> 4
        c[1::2] = packed & 0xF
        return c[:n]
    return {"pack_nibbles": pack_nibbles, "unpack_codes": unpack_codes}


def _k15_planes_neighbours_swapped():
    # consistent on both sides: elements 2j and 2j+1 trade places in the planes
    pack, unpack = O.pack_k15_planes, O.unpack_k15_planes

    def swap(m, n):
        g = np.zeros(-(-n // 32) * 32, dtype=np.uint32)
        g[:n] = m
        return g.reshape(-1, 2)[:, ::-1].reshape(-1)

    return {"pack_k15_planes": lambda raw7: pack(swap(raw7, raw7.size)),
            "unpack_k15_planes": lambda pa, pb, pc, n: swap(unpack(pa, pb, pc, -(-n // 32) * 32),
                                                            -(-n // 32) * 32)[:n]}


def _k15_tail_bits_reversed():
    # consistent on both sides: bit b of a tail element goes to byte 4 (6 - b) + i
    # instead of byte 4 b + i, so everything still round-trips
    def pack(raw7):
        n = raw7.size
        groups = -(-n // 32)
        m = np.zeros(groups * 32, dtype=np.uint32)
        m[:n] = raw7
        m = m.reshape(groups, 32)
        j = np.arange(28)
        tail_bit = (m[:, 28 + (j % 4)] >> (6 - j // 4)) & 1
        mb = (m[:, :28] | (tail_bit << 7)).astype(np.uint8)
        return mb[:, :16].reshape(-1).copy(), mb[:, 16:24].reshape(-1).copy(), mb[:, 24:28].reshape(-1).copy()

    def unpack(pa, pb, pc, n):
        groups = -(-n // 32)
        mb = np.concatenate([pa[:16 * groups].reshape(groups, 16), pb[:8 * groups].reshape(groups, 8),
                             pc[:4 * groups].reshape(groups, 4)], axis=1).astype(np.uint32)
        tail = np.zeros((groups, 4), dtype=np.uint32)
        for b in range(7):
            tail |= ((mb[:, 4 * (6 - b):4 * (6 - b) + 4] >> 7) & 1) << b
        return np.concatenate([mb & 0x7F, tail], axis=1).reshape(-1)[:n].astype(np.uint32)

    return {"pack_k15_planes": pack, "unpack_k15_planes": unpack}


def _index_counts_at_or_below():
    return {"escape_index": lambda pos, bounds: np.searchsorted(pos, bounds, side="right").astype(np.uint32)}


def _k15_escape_keeps_symbol_only():
    orig = O.encode

    def encode(w, scheme, N=None, K=None):
        c = orig(w, scheme, N, K)
        if scheme == O.K15:
            c.esc_val = (c.esc_val >> 7).astype(np.uint16)
        return c
    return {"encode": encode}


def _decode_rows_ignores_escapes():
    orig = O.decode_rows

    def decode_rows(c, rows):
        out = orig(c, rows)
        shift = 8 if c.scheme == O.BYTESPLIT else 7
        for j, r in enumerate(np.asarray(rows)):
            a = int(r) * c.K
            for e in range(int(c.row_index[r]), int(c.row_index[r + 1])):
                p = int(c.esc_pos[e]) - a
                out[j, p] &= (1 << shift) - 1
        return out
    return {"decode_rows": decode_rows}


def _accounting_without_table():
    return {"entropy_bpw": lambda scheme, n, E: 4 + O.RAW_BITS[scheme] + E * O.SYM_BITS[scheme] / n}


def _accounting_with_positions():
    return {"entropy_bpw": lambda scheme, n, E: (4 + O.RAW_BITS[scheme] +
                                                  (E * (O.SYM_BITS[scheme] + 32) +
                                                   O.TABLE_SIZE * O.SYM_BITS[scheme]) / n)}


def _reduction_as_fraction_kept():
    return {"reduction_pct": lambda bpw: 100.0 * bpw / 16.0}


def _gemv_in_fp32():
    def gemv(w_bits, x_bits):
        W = O.bf16_to_f64(w_bits).astype(np.float32)
        X = O.bf16_to_f64(x_bits).astype(np.float32)
        return (X @ W.T).astype(np.float64)
    return {"gemv": gemv}


def _gemv_weight_read_as_k_by_n():
    def gemv(w_bits, x_bits):
        W = O.bf16_to_f64(w_bits)
        X = O.bf16_to_f64(x_bits)
        # the row-major buffer of W[N, K] read as W[K, N]
        return X @ W.reshape(W.shape[1], W.shape[0])
    return {"gemv": gemv}


def _bits9_msb_first():
    def pack_bits9(vals):
        vals = np.asarray(vals, dtype=np.uint32)
        bits = ((vals[:, None] >> np.arange(8, -1, -1, dtype=np.uint32)) & 1).astype(np.uint8).reshape(-1)
        out = np.zeros(-(-bits.size // 8), dtype=np.uint8)
        if bits.size:
            padded = np.zeros(out.size * 8, dtype=np.uint8)
            padded[: bits.size] = bits
            out = np.packbits(padded.reshape(-1, 8), axis=1, bitorder="little").reshape(-1)
        return out

    def unpack_bits9(buf, count):
        bits = np.unpackbits(np.asarray(buf, dtype=np.uint8), bitorder="little")[: 9 * count]
        w = np.arange(8, -1, -1, dtype=np.uint32)
        return (bits.reshape(count, 9).astype(np.uint32) << w).sum(axis=1).astype(np.uint32)
    return {"pack_bits9": pack_bits9, "unpack_bits9": unpack_bits9}


def _payload_checksum_unchecked():
    orig_crc = O.zlib.crc32

    class Z:
        @staticmethod
        def crc32(data):
            # header checksums stay; a payload is any buffer longer than a header
            return 0 if len(data) > 92 else orig_crc(data)
    return {"zlib": Z}


def _compact_k15_escape_without_mantissa():
    orig = O._deserialize_compact

    def _deserialize_compact(buf, scheme, N, K, E, table, plen, pcrc):
        c = orig(buf, scheme, N, K, E, table, plen, pcrc)
        if scheme == O.K15:
            c.esc_val = (c.esc_val & 0xFF80).astype(np.uint16)
        return c
    return {"_deserialize_compact": _deserialize_compact}


def _compact_tile_counts_cumulative():
    # consistent on both sides: the counts section holds each tile's running
    # total (escapes up to the tile's end) instead of the tile's own count
    orig_ser, orig_des = O.serialize_compact, O._deserialize_compact

    def serialize_compact(c):
        saved = c.tile_index
        try:
            # diff of this index is saved[1:], the running totals
            c.tile_index = np.concatenate([[0], np.cumsum(saved[1:].astype(np.int64))]).astype(np.uint32)
            return orig_ser(c)
        finally:
            c.tile_index = saved

    def _deserialize_compact(buf, scheme, N, K, E, table, plen, pcrc):
        off = O.HEADER_BYTES
        for name, size in O.section_sizes_compact(scheme, N, K, E):
            if name == "tile_count":
                break
            off += O._pad(size)
        n_tiles = -(-N * K // O.TILE)
        raw = bytearray(buf)
        running = np.frombuffer(bytes(raw[off: off + 2 * n_tiles]), "<u2").astype(np.int64)
        counts = np.diff(np.concatenate([[0], running]))
        raw[off: off + 2 * n_tiles] = counts.astype("<u2").tobytes()
        payload = bytes(raw[O.HEADER_BYTES:])
        return orig_des(bytes(raw[:O.HEADER_BYTES]) + payload, scheme, N, K, E, table, plen, O.zlib.crc32(payload))
    return {"serialize_compact": serialize_compact, "_deserialize_compact": _deserialize_compact}


def _decode_skips_bytesplit_escapes():
    orig = O.decode

    def decode(c):
        w = orig(c)
        if c.scheme == O.BYTESPLIT and c.E:
            flat = w.reshape(-1)
            flat[c.esc_pos] &= 0x00FF
        return w
    return {"decode": decode}


MUTANTS = {
    "compact_k15_escape_without_mantissa": _compact_k15_escape_without_mantissa,
    "compact_tile_counts_cumulative": _compact_tile_counts_cumulative,
    "decode_skips_bytesplit_escapes": _decode_skips_bytesplit_escapes,
    "tie_break_descending": _tie_break_descending,
    "least_frequent_first": _least_frequent_first,
    "codes_off_by_one": _codes_off_by_one,
    "histogram_without_empty_bins": _histogram_without_empty_bins,
    "k15_symbol_width_8": _k15_symbol_width_8,
    "nibbles_high_first": _nibbles_high_first,
    "k15_planes_neighbours_swapped": _k15_planes_neighbours_swapped,
    "k15_tail_bits_reversed": _k15_tail_bits_reversed,
    "index_counts_at_or_below": _index_counts_at_or_below,
    "k15_escape_keeps_symbol_only": _k15_escape_keeps_symbol_only,
    "decode_rows_ignores_escapes": _decode_rows_ignores_escapes,
    "accounting_without_table": _accounting_without_table,
    "accounting_with_positions": _accounting_with_positions,
    "reduction_as_fraction_kept": _reduction_as_fraction_kept,
    "gemv_in_fp32": _gemv_in_fp32,
    "gemv_weight_read_as_k_by_n": _gemv_weight_read_as_k_by_n,
    "bits9_msb_first": _bits9_msb_first,
    "payload_checksum_unchecked": _payload_checksum_unchecked,
}


def test_unmutated_oracle_passes_every_pin():
    assert _first_failing_pin() is None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    for attr, value in MUTANTS[name]().items():
        monkeypatch.setattr(O, attr, value)
    assert _first_failing_pin() is not None, f"no pin fails with the planted mistake {name}"
