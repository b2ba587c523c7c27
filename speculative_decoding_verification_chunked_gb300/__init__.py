"""Chunked multi-query verification attention for speculative decoding on GB300.

The CUDA library (``libsvx.so``, C ABI in ``include/svx.h``) is loaded lazily
by ``speculative_decoding_verification_chunked_gb300.svx``; importing that
module without a built library raises ImportError.
"""
__all__ = ["svx"]
