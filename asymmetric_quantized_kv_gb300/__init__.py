"""GB300-native decode attention over an asymmetrically quantized KV cache.

The compute lives in libkvq.so (hand-written CUDA for sm_103a behind the C ABI of
include/kvq.h); this package is its ctypes binding plus device-memory plumbing.
Importing the binding fails when the library has not been built.
"""
from . import _binding as binding  # noqa: F401
from ._binding import *  # noqa: F401,F403
from .cache import PagedKVCache, make_config, src_torch_dtype  # noqa: F401
