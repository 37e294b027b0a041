"""Page-locked host buffers for streaming batches to the GPU.

A buffer is anonymous memory mapped with a transparent-huge-page hint,
touched once and registered with the CUDA driver (cudaHostRegister), so the
copy engines read it directly.  Large pages keep the number of translations
a 16 GiB copy walks small; on the Grace hosts this library targets, copies
from such buffers ran at the same ~210 GB/s as ordinary pinned memory and
stalled less often.  Where registration fails, the buffer falls back to
torch's own pinned allocation.
"""
import mmap

import numpy as np


class PinnedBuffer:
    """``tensor`` is a 1-D page-locked host tensor of ``numel`` elements of
    ``dtype`` (a torch dtype); call ``release()`` (or drop the object) when
    no copy from it is still in flight."""

    def __init__(self, torch, numel: int, dtype):
        self._torch = torch
        self._map = None
        self._ptr = None
        itemsize = torch.empty((), dtype=dtype).element_size()
        nbytes = max(int(numel) * itemsize, 1)
        try:
            m = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            if hasattr(mmap, "MADV_HUGEPAGE"):
                m.madvise(mmap.MADV_HUGEPAGE)
            raw = np.frombuffer(m, dtype=np.uint8)
            raw[::4096] = 0  # fault every page in before it is pinned
            ptr = raw.ctypes.data
            err = torch.cuda.cudart().cudaHostRegister(ptr, nbytes, 0)
            if int(err) != 0:
                raise RuntimeError(f"cudaHostRegister: {err}")
            self._map, self._ptr = m, ptr
            self.tensor = torch.frombuffer(m, dtype=dtype, count=int(numel))
        except (RuntimeError, OSError, ValueError, AttributeError):
            self.tensor = torch.empty(int(numel), dtype=dtype).pin_memory()

    def release(self):
        if self._ptr is not None:
            self.tensor = None
            self._torch.cuda.synchronize()
            self._torch.cuda.cudart().cudaHostUnregister(self._ptr)
            self._ptr = None
            try:
                self._map.close()
            except BufferError:
                pass  # a view is still alive; the mapping goes with it
            self._map = None

    def __del__(self):
        try:
            self.release()
        except Exception:
            pass
