"""torch custom op for the plug-and-play attention: ``torch.ops.sage_fp4.attention``.

Importing this module registers the op.  It runs the library's kernels
(quantize Q, K, V, then the FP4 attention) on the current stream through
``sage_fp4.attention``; its fake implementation tells torch.compile and other
tracers the output's shape, dtype and layout without running anything.
"""
from typing import Optional

import torch

from . import sage_fp4 as _S


@torch.library.custom_op("sage_fp4::attention", mutates_args=())
def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
              scale: Optional[float] = None, layout: str = "HND", fmt: str = "nvfp4") -> torch.Tensor:
    """SageAttention3 FP4 attention of bf16 Q, K, V in layout "HND" ([B,H,N,D])
    or "NHD" ([B,N,H,D]) -> new contiguous bf16 O in the same layout; fmt
    "nvfp4" (the method's) or "mxfp4"."""
    return _S.attention(q, k, v, causal=causal, scale=scale, layout=layout, fmt=fmt)


@attention.register_fake
def _attention_fake(q, k, v, causal=False, scale=None, layout="HND", fmt="nvfp4"):
    if layout not in _S.LAYOUTS or fmt not in _S.FORMATS:
        raise ValueError(f"layout must be one of {_S.LAYOUTS}, fmt one of {tuple(_S.FORMATS)}")
    return torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
