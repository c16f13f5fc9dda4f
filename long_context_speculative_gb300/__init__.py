"""GB300-native verification step of retrieval-augmented speculative decoding.

``rapid`` is the binding of librapid.so (verify attention + acceptance, all in
CUDA kernels for sm_103a); ``workloads`` holds the seeded synthetic inputs.
The library is loaded lazily on first use and raises if it is not built.
"""
from . import rapid  # noqa: F401
from .rapid import accept, verify_attn  # noqa: F401

__all__ = ["rapid", "accept", "verify_attn"]
