"""Lossless BF16 weight coding (byte-split and K15) with a fused decode-GEMV for GB300.

The compute path is the CUDA library libwcomp.so (C ABI declared in
include/wcomp.h); ``decode_gemv_sign_gb300.wcomp`` is its Python binding.
``decode_gemv_sign_gb300.synth`` draws seeded synthetic inputs.
"""
__all__ = ["wcomp", "synth"]
