"""GB300-native (sm_103a) SageAttention3 NVFP4 attention forward.

The computing path lives in the CUDA library ``_build/libsagefp4.so`` (C ABI
in ``include/sage_fp4.h``); this package binds it with ctypes.
"""
from .sage_fp4 import (QuantizedQKV, SageFp4Error, attention, attn_fwd, load, quantize_qkv,
                       strerror)

__all__ = ["QuantizedQKV", "SageFp4Error", "attention", "attn_fwd", "load", "quantize_qkv",
           "strerror"]
