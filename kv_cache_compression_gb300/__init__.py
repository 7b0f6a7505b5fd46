"""GB300-native (sm_103a) SnapKV: prefill KV-cache compression and compressed-cache decode attention.

The compute lives in ``libsnapkv.so`` (hand-written CUDA kernels behind the C ABI declared in
``include/snapkv.h``); ``snapkv`` is its thin Python binding.
"""
from . import snapkv  # noqa: F401
from .snapkv import (append, compress, compress_workspace_size, decode_attend,  # noqa: F401
                     decode_workspace_size, kept, make_params, status_string)

__all__ = ["snapkv", "compress", "append", "decode_attend", "kept", "make_params", "compress_workspace_size",
           "decode_workspace_size", "status_string"]
