"""Python binding of the C-ABI library (argument marshalling only).

Every operation runs in the CUDA kernels of libwcomp.so; this module passes
device pointers, sizes and the current CUDA stream through ctypes and turns
status codes into exceptions.  PyTorch is used for device memory and streams.
There is no fallback: if the library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libwcomp.so")

BYTESPLIT = 0
K15 = 1
SCHEMES = {"bytesplit": BYTESPLIT, "byte-split": BYTESPLIT, "k15": K15, BYTESPLIT: BYTESPLIT, K15: K15}

OK, EINVAL, ENOMEM, ECORRUPT, ECUDA, EUNSUPPORTED, ETIMEOUT, EINTERNAL, EBOUNDS = 0, -1, -2, -3, -4, -5, -6, -7, -8


class WcompError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_strerror(status)} ({status})")


class CorruptContainer(WcompError):
    pass


class Info(ctypes.Structure):
    _fields_ = [
        ("scheme", ctypes.c_int32), ("version", ctypes.c_int32),
        ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("n", ctypes.c_int64),
        ("n_escapes", ctypes.c_uint64), ("tile_elems", ctypes.c_uint32), ("n_tiles", ctypes.c_uint32),
        ("table", ctypes.c_uint16 * 15), ("pad_", ctypes.c_uint16),
        ("bytes_codes", ctypes.c_uint64), ("bytes_raw", ctypes.c_uint64), ("bytes_index", ctypes.c_uint64),
        ("bytes_escapes", ctypes.c_uint64), ("serialized_bytes", ctypes.c_uint64),
        ("entropy_bpw", ctypes.c_double), ("physical_bpw", ctypes.c_double),
        ("serialized_compact_bytes", ctypes.c_uint64), ("physical_compact_bpw", ctypes.c_double),
    ]

    def as_dict(self) -> dict:
        d = {k: getattr(self, k) for k, _ in self._fields_ if k not in ("table", "pad_")}
        d["table"] = list(self.table)
        return d


_lib = None
P = ctypes.c_void_p


def lib():
    """Load libwcomp.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    L = ctypes.CDLL(LIB_PATH)
    L.wcomp_encode.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P, ctypes.POINTER(P)]
    L.wcomp_encode_batched.argtypes = [ctypes.POINTER(P), ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int), ctypes.c_int,
                                       P, ctypes.POINTER(P)]
    L.wcomp_encode_hist_grid.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_uint32)]
    L.wcomp_decode.argtypes = [P, P, P]
    L.wcomp_gemv.argtypes = [P, P, ctypes.c_int, P, P]
    L.wcomp_gemv_noalloc.argtypes = [P, P, ctypes.c_int, P, P]
    L.wcomp_gemv_bf16.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_int, P, P]
    L.wcomp_gemv_bf16_batched.argtypes = [ctypes.POINTER(P), ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(P), ctypes.c_int,
                                          ctypes.POINTER(P), ctypes.c_int, P]
    L.wcomp_decode_batched.argtypes = [ctypes.POINTER(P), ctypes.POINTER(P), ctypes.c_int, P]
    L.wcomp_gemv_batched.argtypes = [ctypes.POINTER(P), ctypes.POINTER(P), ctypes.c_int, ctypes.POINTER(P),
                                     ctypes.c_int, P]
    L.wcomp_info.argtypes = [P, ctypes.POINTER(Info)]
    L.wcomp_serialize.argtypes = [P, P, ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64), P]
    L.wcomp_serialize_compact.argtypes = [P, P, ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64), P]
    L.wcomp_deserialize.argtypes = [P, ctypes.c_uint64, P, ctypes.POINTER(P)]
    L.wcomp_free.argtypes = [P, P]
    L.wcomp_free.restype = None
    L.wcomp_strerror.argtypes = [ctypes.c_int]
    L.wcomp_strerror.restype = ctypes.c_char_p
    L.wcomp_version.argtypes = []
    L.wcomp_device_check.argtypes = [P]
    L.wcomp_device_check.restype = ctypes.c_int
    L.wcomp_debug_skip_first_copy.argtypes = [ctypes.c_int]
    L.wcomp_debug_skip_first_copy.restype = ctypes.c_int
    L.wcomp_launch_count.argtypes = []
    L.wcomp_launch_count.restype = ctypes.c_uint64
    for name in ("wcomp_encode", "wcomp_encode_batched", "wcomp_encode_hist_grid", "wcomp_decode", "wcomp_gemv", "wcomp_gemv_noalloc",
                 "wcomp_gemv_bf16", "wcomp_gemv_bf16_batched",
                 "wcomp_decode_batched",
                 "wcomp_gemv_batched", "wcomp_info", "wcomp_serialize", "wcomp_serialize_compact",
                 "wcomp_deserialize", "wcomp_version", "wcomp_debug_skip_first_copy"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _strerror(s: int) -> str:
    try:
        return lib().wcomp_strerror(s).decode()
    except Exception:  # pragma: no cover
        return "error"


def _check(status: int, what: str):
    if status == ECORRUPT:
        raise CorruptContainer(status, what)
    if status != OK:
        raise WcompError(status, what)


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _bits16(t: torch.Tensor, what: str) -> torch.Tensor:
    """A contiguous CUDA tensor of 16-bit BF16 bit patterns (bf16, int16 or uint16)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{what} must hold BF16 bits (bfloat16, int16 or uint16), got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t


class Container:
    """An encoded tensor living on the GPU (owned by the library)."""

    def __init__(self, handle: int, shape=None):
        self._h = handle
        self._info = None
        self._shape = tuple(shape) if shape is not None else None  # (N, K) when the caller knows it

    @property
    def handle(self) -> int:
        if not self._h:
            raise ValueError("container was freed")
        return self._h

    def info(self) -> dict:
        if self._info is None:
            inf = Info()
            _check(lib().wcomp_info(P(self.handle), ctypes.byref(inf)), "wcomp_info")
            self._info = inf.as_dict()
        return self._info

    @property
    def shape(self) -> tuple:
        """(N, K), without a description call when the shape is known from the encode."""
        if self._shape is None:
            inf = self.info()
            self._shape = (inf["N"], inf["K"])
        return self._shape

    @property
    def N(self) -> int:
        return self.shape[0]

    @property
    def K(self) -> int:
        return self.shape[1]

    @property
    def scheme(self) -> int:
        return self.info()["scheme"]

    def free(self, stream=None):
        if self._h:
            lib().wcomp_free(P(self._h), P(_stream(stream)))
            self._h = 0

    def __del__(self):
        try:
            if self._h and torch.cuda.is_available():
                self.free()
        except Exception:
            pass


def encode(w: torch.Tensor, scheme, stream=None) -> Container:
    """Encode BF16 weights W[N, K] (a 1-D tensor is one row)."""
    w = _bits16(w, "w")
    N, K = (w.shape[0], w.shape[1]) if w.dim() == 2 else (1, w.numel())
    if w.dim() not in (1, 2):
        raise ValueError("w must be 1-D or 2-D")
    h = P()
    _check(lib().wcomp_encode(P(w.data_ptr()), N, K, SCHEMES[scheme], P(_stream(stream)), ctypes.byref(h)),
           "wcomp_encode")
    return Container(h.value, (N, K))


def encode_batched(ws: Sequence[torch.Tensor], schemes, stream=None) -> List[Container]:
    """Encode several tensors in one batched pass (one host synchronization).

    ``schemes`` is one scheme for all tensors or a sequence with one per tensor.
    """
    n = len(ws)
    if isinstance(schemes, (str, int)):
        schemes = [schemes] * n
    Ns, Ks = [], []
    for w in ws:
        _bits16(w, "w")
        if w.dim() not in (1, 2):
            raise ValueError("w must be 1-D or 2-D")
        Ns.append(w.shape[0] if w.dim() == 2 else 1)
        Ks.append(w.shape[1] if w.dim() == 2 else w.numel())
    outs = (P * n)()
    _check(lib().wcomp_encode_batched(_ptr_array([w.data_ptr() for w in ws]), (ctypes.c_int64 * n)(*Ns),
                                      (ctypes.c_int64 * n)(*Ks), (ctypes.c_int * n)(*[SCHEMES[x] for x in schemes]),
                                      n, P(_stream(stream)), outs), "wcomp_encode_batched")
    return [Container(outs[i], (Ns[i], Ks[i])) for i in range(n)]


def decode(c: Container, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Exact BF16 bits of W[N, K] as an int16 tensor (``out`` if given)."""
    inf = c.info()
    if out is None:
        out = torch.empty((inf["N"], inf["K"]), dtype=torch.int16, device="cuda")
    out = _bits16(out, "out")
    if out.numel() != inf["n"]:
        raise ValueError("out has the wrong size")
    _check(lib().wcomp_decode(P(c.handle), P(out.data_ptr()), P(_stream(stream))), "wcomp_decode")
    return out


def gemv(c: Container, x: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y[B, N] (fp32) = x[B, K] @ W.T with W decoded in registers."""
    x = _bits16(x, "x")
    N, K = c.shape
    B = x.shape[0] if x.dim() == 2 else 1
    if x.numel() != B * K:
        raise ValueError("x has the wrong size")
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device="cuda")
    if y.dtype != torch.float32 or not y.is_contiguous() or y.numel() != B * N:
        raise ValueError("y must be a contiguous float32 tensor of B*N elements")
    _check(lib().wcomp_gemv(P(c.handle), P(x.data_ptr()), B, P(y.data_ptr()), P(_stream(stream))), "wcomp_gemv")
    return y


def gemv_noalloc(c: Container, x: torch.Tensor, y: torch.Tensor, stream=None) -> torch.Tensor:
    """wcomp_gemv without any device allocation by the library.

    For callers that cannot let a library allocate device memory (a fixed
    memory budget, or no implicit synchronisation from cudaMalloc / cudaFree).
    ``y`` must be supplied by the caller.  Calls share one small static device
    array: do not let two of them run at the same time on different streams.
    """
    x = _bits16(x, "x")
    N, K = c.shape
    B = x.shape[0] if x.dim() == 2 else 1
    if x.numel() != B * K:
        raise ValueError("x has the wrong size")
    if y.dtype != torch.float32 or not y.is_contiguous() or y.numel() != B * N:
        raise ValueError("y must be a contiguous float32 tensor of B*N elements")
    _check(lib().wcomp_gemv_noalloc(P(c.handle), P(x.data_ptr()), B, P(y.data_ptr()), P(_stream(stream))),
           "wcomp_gemv_noalloc")
    return y


def gemv_bf16(w: torch.Tensor, x: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Plain BF16 GEMV (the comparison kernel)."""
    w = _bits16(w, "w")
    x = _bits16(x, "x")
    N, K = (w.shape[0], w.shape[1]) if w.dim() == 2 else (1, w.numel())
    B = x.shape[0] if x.dim() == 2 else 1
    if x.numel() != B * K:
        raise ValueError("x has the wrong size")
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device="cuda")
    _check(lib().wcomp_gemv_bf16(P(w.data_ptr()), N, K, P(x.data_ptr()), B, P(y.data_ptr()), P(_stream(stream))),
           "wcomp_gemv_bf16")
    return y


def gemv_bf16_batched(ws: Sequence[torch.Tensor], xs: Sequence[torch.Tensor],
                      ys: Optional[List[torch.Tensor]] = None, stream=None):
    """Plain BF16 GEMV over several weight tensors in one launch."""
    B = xs[0].shape[0] if xs[0].dim() == 2 else 1
    Ns, Ks = [], []
    for w, x in zip(ws, xs):
        _bits16(w, "w")
        _bits16(x, "x")
        N, K = (w.shape[0], w.shape[1]) if w.dim() == 2 else (1, w.numel())
        if x.numel() != B * K:
            raise ValueError("x has the wrong size")
        Ns.append(N)
        Ks.append(K)
    if ys is None:
        ys = [torch.empty((B, N), dtype=torch.float32, device="cuda") for N in Ns]
    n_arr = (ctypes.c_int64 * len(ws))(*Ns)
    k_arr = (ctypes.c_int64 * len(ws))(*Ks)
    _check(lib().wcomp_gemv_bf16_batched(_ptr_array([w.data_ptr() for w in ws]), n_arr, k_arr,
                                         _ptr_array([x.data_ptr() for x in xs]), B,
                                         _ptr_array([y.data_ptr() for y in ys]), len(ws), P(_stream(stream))),
           "wcomp_gemv_bf16_batched")
    return ys


def _ptr_array(ptrs: Sequence[int]):
    arr = (P * len(ptrs))()
    for i, p in enumerate(ptrs):
        arr[i] = p
    return arr


def decode_batched(cs: Sequence[Container], outs: Optional[List[torch.Tensor]] = None, stream=None):
    if outs is None:
        outs = [torch.empty((c.N, c.K), dtype=torch.int16, device="cuda") for c in cs]
    for c, o in zip(cs, outs):
        _bits16(o, "out")
        N, K = c.shape
        if o.numel() != N * K:
            raise ValueError("output has the wrong size")
    _check(lib().wcomp_decode_batched(_ptr_array([c.handle for c in cs]), _ptr_array([o.data_ptr() for o in outs]),
                                      len(cs), P(_stream(stream))), "wcomp_decode_batched")
    return outs


def gemv_batched(cs: Sequence[Container], xs: Sequence[torch.Tensor], ys: Optional[List[torch.Tensor]] = None,
                 stream=None):
    B = xs[0].shape[0] if xs[0].dim() == 2 else 1
    for c, x in zip(cs, xs):
        _bits16(x, "x")
        if x.numel() != B * c.K:
            raise ValueError("x has the wrong size")
    if ys is None:
        ys = [torch.empty((B, c.N), dtype=torch.float32, device="cuda") for c in cs]
    _check(lib().wcomp_gemv_batched(_ptr_array([c.handle for c in cs]), _ptr_array([x.data_ptr() for x in xs]), B,
                                    _ptr_array([y.data_ptr() for y in ys]), len(cs), P(_stream(stream))),
           "wcomp_gemv_batched")
    return ys


def serialize(c: Container, stream=None, compact: bool = False) -> bytes:
    """Container bytes: format version 1, or version 2 (compact) with compact=True."""
    fn = lib().wcomp_serialize_compact if compact else lib().wcomp_serialize
    name = "wcomp_serialize_compact" if compact else "wcomp_serialize"
    n = ctypes.c_uint64()
    _check(fn(P(c.handle), None, 0, ctypes.byref(n), P(_stream(stream))), name)
    buf = ctypes.create_string_buffer(n.value)
    _check(fn(P(c.handle), buf, n.value, ctypes.byref(n), P(_stream(stream))), name)
    return buf.raw[: n.value]


def deserialize(data: bytes, stream=None) -> Container:
    h = P()
    buf = ctypes.create_string_buffer(bytes(data), len(data))
    _check(lib().wcomp_deserialize(buf, len(data), P(_stream(stream)), ctypes.byref(h)), "wcomp_deserialize")
    return Container(h.value)


def version() -> int:
    return lib().wcomp_version()


def device_check(stream=None) -> None:
    """Raise if a kernel on this device reported a timed-out wait (clears the report)."""
    _check(lib().wcomp_device_check(P(_stream(stream))), "wcomp_device_check")


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().wcomp_launch_count())
