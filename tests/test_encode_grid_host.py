"""The encoder's histogram grid keeps every 16-bit counter half below 65,536.

hist_kernel counts into 16-bit halves of shared-memory words; each half
collects one lane of each of the block's 8 warps, and work is dealt out in
8-element chunks (thread t of block b takes chunks b*256 + t, + 256*blocks,
...).  The worst case for a half is a constant tensor: every element lands in
one bin.  This test asks the library how it sizes the grid
(wcomp_encode_hist_grid, host-side, no GPU) and simulates that chunk
distribution exactly, for single tensors and for batches where a small tensor
shares the grid with a very large one (so its share of blocks is at the
lower bound).  No GPU is needed.
"""
import ctypes

import numpy as np
import pytest

from decode_gemv_sign_gb300 import wcomp

THREADS, WARPS, CHUNK, HALF_MAX = 256, 8, 8, 65535


@pytest.fixture(scope="module")
def lib():
    from decode_gemv_sign_gb300 import build

    build.build()
    return wcomp.lib()


def grid(lib, ns, sms=152):
    arr = (ctypes.c_uint64 * len(ns))(*ns)
    out = (ctypes.c_uint32 * len(ns))()
    assert lib.wcomp_encode_hist_grid(arr, len(ns), sms, out) == wcomp.OK
    return list(out)


def worst_half(n: int, blocks: int) -> int:
    """Largest number of elements one counter half receives when all n elements share a symbol."""
    chunks = -(-n // CHUNK)
    stride = blocks * THREADS
    # elements thread i handles: its chunks i, i + stride, ...; the last chunk of the tensor may be short
    i = np.arange(stride, dtype=np.int64)
    nch = np.where(i < chunks, (chunks - 1 - i) // stride + 1, 0)
    last = i + (nch - 1) * stride  # index of the thread's last chunk
    elems = nch * CHUNK - np.where((nch > 0) & (last == chunks - 1), chunks * CHUNK - n, 0)
    # thread i = blk * 256 + tid; lane = tid % 32; half = (lane % 16, lane // 16); 8 warps share a half
    tid = i % THREADS
    blk = i // THREADS
    half = (tid % 32)
    key = blk * 32 + half
    sums = np.bincount(key, weights=elems, minlength=blocks * 32)
    return int(sums.max())


def test_single_tensors_stay_below_the_limit(lib):
    sms = 152
    for n in [1, 7, 8, 9, 2047, 2048, 2049, 8191 * 256, 512 * 8191, 4_193_792, 6_290_688, 931_021_824,
              1 << 31, 2_147_483_648 + 12345, 3_000_000_000, (1 << 32) - 1]:
        (b,) = grid(lib, [n], sms)
        assert 1 <= b <= -(-(-(-n // CHUNK)) // THREADS)
        assert worst_half(n, b) <= HALF_MAX, (n, b)


def test_small_tensors_in_huge_batches_stay_below_the_limit(lib):
    """The cases that wrapped with the element-count bound: a tensor whose share of a
    large batch drops its block count to the counter bound."""
    rng = np.random.default_rng(0)
    smalls = [4_193_792, 6_290_688, 512 * 8191, 1023 * 256 * 8, 1023 * 256 * 8 + 1, 2 * 1023 * 256 * 8 - 8,
              931_021_824] + [int(v) for v in rng.integers(1, 1 << 27, size=40)]
    for small in smalls:
        for big in [2_000_000_000, (1 << 32) - 1]:
            b_small, _ = grid(lib, [small, big])
            assert worst_half(small, b_small) <= HALF_MAX, (small, big, b_small)


def test_the_old_element_bound_would_wrap():
    """The bound this replaces (8191 elements per thread on average) lets a half reach 65,536."""
    n = 512 * 8191
    blocks = -(-n // (8191 * 256))
    assert worst_half(n, blocks) == 65536


def test_grid_rejects_bad_arguments(lib):
    out = (ctypes.c_uint32 * 1)()
    arr = (ctypes.c_uint64 * 1)(0)
    assert lib.wcomp_encode_hist_grid(arr, 1, 152, out) == wcomp.EINVAL
    arr = (ctypes.c_uint64 * 1)(1 << 32)
    assert lib.wcomp_encode_hist_grid(arr, 1, 152, out) == wcomp.EINVAL
    assert lib.wcomp_encode_hist_grid(None, 1, 152, out) == wcomp.EINVAL
    arr = (ctypes.c_uint64 * 1)(100)
    assert lib.wcomp_encode_hist_grid(arr, 0, 152, out) == wcomp.EINVAL
    assert lib.wcomp_encode_hist_grid(arr, 1, 0, out) == wcomp.EINVAL
