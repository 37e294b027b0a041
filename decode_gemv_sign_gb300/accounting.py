"""Algorithmic bytes per launch: the minimum traffic each operation implies.

Byte counts from a container's description (wcomp_info as a dict): the code
stream, the raw low bytes or K15 mantissa planes, the escape index the
operation uses (per tile for decode, per row for the GEMV), the escape
positions (4 bytes) and values (the whole 16-bit word, as the device
container keeps them for both schemes), plus what the operation writes
(decode: 2 bytes per element; GEMV: x read once, y written as fp32).  These are the numerators of the roofline fractions.
"""


def container_read_bytes(info: dict, part: str) -> int:
    """Bytes a decode ("decode") or fused GEMV ("gemv") must read from a container."""
    n_tiles_b = 4 * (info["n_tiles"] + 1)
    rows_b = 4 * (info["N"] + 1)
    E = info["n_escapes"]
    val = 2 * E
    streams = info["bytes_codes"] + info["bytes_raw"]
    if part == "decode":
        return streams + n_tiles_b + 4 * E + val
    return streams + rows_b + 4 * E + val


def encode_bytes(info: dict) -> int:
    # read the source once, write the container once
    return 2 * info["n"] + info["serialized_bytes"] - 96


def decode_bytes(info: dict) -> int:
    return container_read_bytes(info, "decode") + 2 * info["n"]


def gemv_bytes(info: dict, B: int) -> int:
    return container_read_bytes(info, "gemv") + 2 * B * info["K"] + 4 * B * info["N"]


def plain_bytes(N: int, K: int, B: int) -> int:
    return 2 * N * K + 2 * B * K + 4 * B * N
