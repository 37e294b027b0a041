"""The C-ABI library loads and exports every entry point that include/wcomp.h
declares; host-side checks (argument errors, corrupt serialized containers)
run without a GPU and agree with the CPU oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

from decode_gemv_sign_gb300 import synth, wcomp
from oracle import wcomp_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wcomp.h")


@pytest.fixture(scope="module")
def lib():
    from decode_gemv_sign_gb300 import build

    build.build()
    return wcomp.lib()


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"WCOMP_API\s+[\w\s\*]+?\b(wcomp_\w+)\s*\(", src)))


def test_header_declares_the_api():
    names = declared()
    for n in ["wcomp_encode", "wcomp_encode_batched", "wcomp_decode", "wcomp_gemv", "wcomp_gemv_noalloc",
              "wcomp_gemv_bf16", "wcomp_gemv_bf16_batched",
              "wcomp_decode_batched", "wcomp_launch_count", "wcomp_device_check",
              "wcomp_gemv_batched", "wcomp_info", "wcomp_serialize", "wcomp_deserialize", "wcomp_free",
              "wcomp_strerror", "wcomp_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared():
        assert hasattr(lib, n), n
    assert lib.wcomp_version() == 1
    assert lib.wcomp_strerror(-3) == b"corrupt container"


def test_argument_errors_without_gpu(lib):
    h = ctypes.c_void_p()
    assert lib.wcomp_encode(None, 4, 4, 0, None, ctypes.byref(h)) == wcomp.EINVAL
    assert lib.wcomp_encode(ctypes.c_void_p(256), 4, 4, 7, None, ctypes.byref(h)) == wcomp.EINVAL
    assert lib.wcomp_encode(ctypes.c_void_p(256), 0, 4, 0, None, ctypes.byref(h)) == wcomp.EINVAL
    assert lib.wcomp_encode(ctypes.c_void_p(256), 1 << 20, 1 << 12, 0, None, ctypes.byref(h)) == wcomp.EUNSUPPORTED
    assert lib.wcomp_encode(ctypes.c_void_p(256), 4, 4, 0, None, None) == wcomp.EINVAL
    assert lib.wcomp_info(None, None) == wcomp.EINVAL
    assert lib.wcomp_decode(None, None, None) == wcomp.EINVAL
    assert lib.wcomp_gemv(None, None, 1, None, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_bf16(ctypes.c_void_p(256), 4, 4, ctypes.c_void_p(256), 0, ctypes.c_void_p(256),
                               None) == wcomp.EINVAL
    assert lib.wcomp_gemv_bf16(ctypes.c_void_p(256), 4, 4, ctypes.c_void_p(256), 17, ctypes.c_void_p(256),
                               None) == wcomp.EINVAL
    lib.wcomp_free(None, None)  # no-op


def _ptrs(*vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_batched_and_remaining_argument_errors_without_gpu(lib):
    """Every entry point rejects bad arguments on the host, before any CUDA call."""
    h = ctypes.c_void_p()
    P = ctypes.c_void_p
    n1 = (ctypes.c_int64 * 1)(4)
    k1 = (ctypes.c_int64 * 1)(4)
    s1 = (ctypes.c_int * 1)(0)
    ok = _ptrs(256)
    # batched encode: null arrays, empty batch, null entry, bad scheme, zero size, null output
    assert lib.wcomp_encode_batched(None, n1, k1, s1, 1, None, ctypes.byref(h)) == wcomp.EINVAL
    assert lib.wcomp_encode_batched(ok, n1, k1, s1, 0, None, ctypes.byref(h)) == wcomp.EINVAL
    assert lib.wcomp_encode_batched(ok, n1, k1, s1, 1, None, None) == wcomp.EINVAL
    # batched decode and GEMV: null arrays and empty batches
    assert lib.wcomp_decode_batched(None, ok, 1, None) == wcomp.EINVAL
    assert lib.wcomp_decode_batched(ok, None, 1, None) == wcomp.EINVAL
    assert lib.wcomp_decode_batched(ok, ok, 0, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_batched(None, ok, 1, ok, 1, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_batched(ok, ok, 1, ok, 0, None) == wcomp.EINVAL
    # containers' GEMV with a null entry inside the arrays
    assert lib.wcomp_gemv_batched(_ptrs(None), ok, 1, ok, 1, None) == wcomp.EINVAL
    # no-allocation GEMV: null pointers and B outside 1..16
    assert lib.wcomp_gemv_noalloc(None, P(256), 1, P(256), None) == wcomp.EINVAL
    # plain GEMV, batched: B outside 1..16, zero sizes, null entries, rows beyond 2^31
    for B in (0, 17):
        assert lib.wcomp_gemv_bf16_batched(ok, n1, k1, ok, B, ok, 1, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_bf16_batched(ok, (ctypes.c_int64 * 1)(0), k1, ok, 1, ok, 1, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_bf16_batched(ok, n1, (ctypes.c_int64 * 1)(-1), ok, 1, ok, 1, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_bf16_batched(_ptrs(None), n1, k1, ok, 1, ok, 1, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_bf16_batched(ok, n1, k1, ok, 1, _ptrs(None), 1, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_bf16_batched(ok, n1, k1, ok, 1, ok, 0, None) == wcomp.EINVAL
    assert lib.wcomp_gemv_bf16(P(256), 1 << 31, 4, P(256), 1, P(256), None) == wcomp.EUNSUPPORTED
    assert lib.wcomp_gemv_bf16(P(256), 4, 0, P(256), 1, P(256), None) == wcomp.EINVAL
    # (de)serialization: null container, null length, null buffer, null output
    n = ctypes.c_uint64()
    assert lib.wcomp_serialize(None, None, 0, ctypes.byref(n), None) == wcomp.EINVAL
    assert lib.wcomp_serialize_compact(None, None, 0, ctypes.byref(n), None) == wcomp.EINVAL
    assert lib.wcomp_deserialize(None, 96, None, ctypes.byref(h)) == wcomp.EINVAL
    assert lib.wcomp_deserialize(ctypes.create_string_buffer(96), 96, None, None) == wcomp.EINVAL
    assert lib.wcomp_info(P(256), None) == wcomp.EINVAL


def test_debug_hook_is_inert_in_the_release_build(lib):
    # the bounded-wait test hook exists in every build but acts only in debug
    # builds; the release library answers without touching a device
    assert lib.wcomp_debug_skip_first_copy(1) == wcomp.EUNSUPPORTED
    assert lib.wcomp_debug_skip_first_copy(0) == wcomp.EUNSUPPORTED


def test_every_status_has_its_own_message(lib):
    codes = [wcomp.OK, wcomp.EINVAL, wcomp.ENOMEM, wcomp.ECORRUPT, wcomp.ECUDA, wcomp.EUNSUPPORTED, wcomp.ETIMEOUT,
             wcomp.EINTERNAL, wcomp.EBOUNDS]
    msgs = [lib.wcomp_strerror(c) for c in codes]
    assert all(msgs) and len(set(msgs)) == len(codes)
    assert lib.wcomp_strerror(-99) == b"unknown status"
    # the header's enum and the binding agree
    src = open(HEADER).read()
    enum = dict((k, int(v)) for k, v in re.findall(r"WCOMP_(OK|E[A-Z]+)\s*=\s*(-?\d+)", src))
    assert enum == {"OK": 0, "EINVAL": -1, "ENOMEM": -2, "ECORRUPT": -3, "ECUDA": -4, "EUNSUPPORTED": -5,
                    "ETIMEOUT": -6, "EINTERNAL": -7, "EBOUNDS": -8}
    assert [enum[k] for k in ("OK", "EINVAL", "ENOMEM", "ECORRUPT", "ECUDA", "EUNSUPPORTED", "ETIMEOUT",
                              "EINTERNAL", "EBOUNDS")] == codes


def _deser_status(lib, buf: bytes) -> int:
    h = ctypes.c_void_p()
    b = ctypes.create_string_buffer(buf, len(buf))
    return lib.wcomp_deserialize(b, len(buf), None, ctypes.byref(h))


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_host_validation_matches_oracle(lib, scheme):
    """Corrupt bytes are rejected on the host (before any device call); intact
    oracle containers pass validation (the call then proceeds to the device)."""
    w = synth.gen_weights_np(synth.WeightSpec("t", 16, 1000, "t4", 0.02, 0.02, "normal", 1.0, seed=5))
    buf = bytearray(O.serialize(O.encode(w, scheme)))
    ok = _deser_status(lib, bytes(buf))
    assert ok != wcomp.ECORRUPT  # OK with a GPU present, a CUDA error without one
    rng = np.random.default_rng(1)
    for off in [0, 4, 6, 8, 24, 32, 40, 72, 80, 92] + list(rng.integers(96, len(buf), size=16)):
        bad = bytearray(buf)
        bad[off] ^= 0x04
        with pytest.raises(O.CorruptContainer):
            O.deserialize(bytes(bad))
        assert _deser_status(lib, bytes(bad)) == wcomp.ECORRUPT
    assert _deser_status(lib, bytes(buf[:-32])) == wcomp.ECORRUPT
    assert _deser_status(lib, bytes(buf[:40])) == wcomp.ECORRUPT


def _recrc(buf: bytearray):
    import struct
    import zlib
    payload = bytes(buf[96:])
    struct.pack_into("<I", buf, 80, zlib.crc32(payload))
    struct.pack_into("<I", buf, 92, zlib.crc32(bytes(buf[:92])))


def test_semantic_corruption_with_valid_checksums(lib):
    """Checksums re-computed after tampering: the structural checks still catch it."""
    import struct
    w = synth.gen_weights_np(synth.WeightSpec("t", 8, 4096, "t4", 0.02, 0.02, "normal", 1.0, seed=6))
    c = O.encode(w, O.BYTESPLIT)
    assert c.E >= 2
    buf = bytearray(O.serialize(c))
    sizes = O.section_sizes(c.scheme, c.N, c.K, c.E)
    off = {}
    p = 96
    for name, sz in sizes:
        off[name] = p
        p += O._pad(sz)
    # 1. escape positions out of order
    bad = bytearray(buf)
    a, b = struct.unpack_from("<II", bad, off["esc_pos"])
    struct.pack_into("<II", bad, off["esc_pos"], b, a)
    _recrc(bad)
    assert _deser_status(lib, bytes(bad)) == wcomp.ECORRUPT
    # 2. a position beyond n
    bad = bytearray(buf)
    struct.pack_into("<I", bad, off["esc_pos"] + 4 * (c.E - 1), c.n + 5)
    _recrc(bad)
    assert _deser_status(lib, bytes(bad)) == wcomp.ECORRUPT
    # 3. tile index disagreeing with the positions
    bad = bytearray(buf)
    struct.pack_into("<I", bad, off["tile_index"] + 4, 0xFFFF)
    _recrc(bad)
    assert _deser_status(lib, bytes(bad)) == wcomp.ECORRUPT
    # 4. a duplicate table symbol
    bad = bytearray(buf)
    t0 = struct.unpack_from("<H", bad, 40)[0]
    struct.pack_into("<H", bad, 42, t0)
    _recrc(bad)
    assert _deser_status(lib, bytes(bad)) == wcomp.ECORRUPT


@pytest.mark.parametrize("scheme", O.SCHEMES)
def test_host_validation_of_compact_form(lib, scheme):
    """The compact form (version 2) is validated on the host like version 1:
    intact oracle bytes pass, flipped bits and count mismatches with re-computed
    checksums are rejected before any device call."""
    import struct
    w = synth.gen_weights_np(synth.WeightSpec("t", 8, 4096, "t4", 0.02, 0.02, "normal", 1.0, seed=7))
    c = O.encode(w, scheme)
    assert c.E >= 2
    buf = bytearray(O.serialize_compact(c))
    assert _deser_status(lib, bytes(buf)) != wcomp.ECORRUPT
    rng = np.random.default_rng(2)
    for off in [4, 8, 24, 72, 80] + list(rng.integers(96, len(buf), size=12)):
        bad = bytearray(buf)
        bad[off] ^= 0x10
        assert _deser_status(lib, bytes(bad)) == wcomp.ECORRUPT
    assert _deser_status(lib, bytes(buf[:-32])) == wcomp.ECORRUPT
    sizes = O.section_sizes_compact(c.scheme, c.N, c.K, c.E)
    off = {}
    p = 96
    for name, sz in sizes:
        off[name] = p
        p += O._pad(sz)
    # an escape code cleared: fewer codes 15 than E
    bad = bytearray(buf)
    i = int(c.esc_pos[0])
    bad[off["codes"] + i // 2] &= 0x0F if i % 2 else 0xF0
    _recrc(bad)
    assert _deser_status(lib, bytes(bad)) == wcomp.ECORRUPT
    # a tile count changed while E stays the same
    bad = bytearray(buf)
    t0 = struct.unpack_from("<H", bad, off["tile_count"])[0]
    struct.pack_into("<H", bad, off["tile_count"], t0 + 1)
    struct.pack_into("<H", bad, off["tile_count"] + 2, struct.unpack_from("<H", bad, off["tile_count"] + 2)[0] - 1)
    _recrc(bad)
    assert _deser_status(lib, bytes(bad)) == wcomp.ECORRUPT


def test_info_struct_layout_matches_the_header(tmp_path):
    """The binding's Info mirrors wcomp_info_t field for field: same names in
    the same order, and the C compiler's offsets and size equal ctypes'."""
    import shutil
    import subprocess

    src = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} wcomp_info_t;", src, re.S).group(1)
    names = []
    for decl in re.sub(r"/\*.*?\*/", "", body, flags=re.S).split(";"):
        decl = decl.strip()
        if not decl:
            continue
        for part in decl.split(None, 1)[1].split(","):
            names.append(part.strip().split("[")[0])
    assert names == [f for f, _ in wcomp.Info._fields_]
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    prog = tmp_path / "off.c"
    prog.write_text('#include <stdio.h>\n#include "wcomp.h"\nint main(void){\n' +
                    "".join(f'printf("%zu\\n", offsetof(wcomp_info_t, {n}));\n' for n in names) +
                    'printf("%zu\\n", sizeof(wcomp_info_t)); return 0; }\n')
    exe = tmp_path / "off"
    subprocess.run([cc, "-std=c99", "-I", os.path.dirname(HEADER), str(prog), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [getattr(wcomp.Info, n).offset for n in names] + [ctypes.sizeof(wcomp.Info)]
    assert got == want


def _c_kind(decl: str):
    if "*" in decl:
        return "ptr"
    base = decl.replace("const", "").split()[0]
    return {"int": ("int", 4), "int32_t": ("int", 4), "int64_t": ("int", 8), "uint64_t": ("uint", 8),
            "uint32_t": ("uint", 4)}[base]


def _py_kind(t):
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "ptr"
    return ("int" if t(-1).value < 0 else "uint", ctypes.sizeof(t))


def test_binding_prototypes_match_the_header(lib):
    """Every declared entry point: the binding passes as many arguments as the
    header declares, each a pointer or an integer of the declared width and
    signedness, and reads the declared return type."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = re.findall(r"WCOMP_API\s+([\w\s\*]+?)\s*\b(wcomp_\w+)\s*\(([^)]*)\)\s*;", src)
    assert sorted(name for _, name, _ in protos) == declared()
    for ret, name, params in protos:
        fn = getattr(lib, name)
        params = params.strip()
        want = [] if params in ("", "void") else [_c_kind(p) for p in params.split(",")]
        assert fn.argtypes is not None, name
        assert [_py_kind(t) for t in fn.argtypes] == want, name
        ret = ret.strip()
        if ret == "void":
            assert fn.restype is None, name
        elif "*" in ret:
            assert _py_kind(fn.restype) == "ptr", name
        else:
            assert _py_kind(fn.restype) == _c_kind(ret), name
