"""GB300-native (sm_103a) SageAttention3 NVFP4 attention forward.

The computing path lives in the CUDA library ``_build/libsagefp4.so`` (C ABI
in ``include/sage_fp4.h``); this package binds it with ctypes.
"""
from .sage_fp4 import (HostWorkspace, QuantizedQKV, SageFp4Error, attention, attention_host, attn_fwd,
                       load, quantize_qkv, strerror)

__all__ = ["HostWorkspace", "QuantizedQKV", "SageFp4Error", "attention", "attention_host", "attn_fwd",
           "load", "quantize_qkv", "strerror"]
