"""GB300 (sm_103a) routed-expert MoE decode for GGUF- and NVFP4-quantized expert banks.

The compute lives in the C-ABI library built from ``csrc/`` (see
``include/qre_moe.h``); ``capi`` is its ctypes binding and ``layer.MoeLayer``
a small convenience wrapper that uses torch for device memory and streams.
Importing ``capi`` raises if the library has not been built -- there is no
fallback path.
"""
from .build import lib_path  # noqa: F401
