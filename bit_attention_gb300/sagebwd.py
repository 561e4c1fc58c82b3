"""Thin Python binding of the SageBwd C ABI in ``include/sagebwd.h``.

SageBwd is the 8-bit attention for training of the SageAttention3 article
("INT8 attention for training"): forward and backward with six of the seven
products in INT8 and dP = dO V^T in FP16.  Argument marshalling only: every
step runs in the CUDA kernels of ``_build/libsagefp4.so``; there is no
fallback, and a failed call raises.

``sagebwd_*`` functions mirror the C entry points and take raw pointers;
``forward``, ``backward`` and ``attention`` (a ``torch.autograd.Function``)
are the torch-tensor conveniences built on them.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import sage_fp4 as _fp4
from .sage_fp4 import EINVAL, OK, SageFp4Error

_HEADER = os.path.join(os.path.dirname(_fp4._HEADER), "sagebwd.h")
WS_FIELDS = 17
WS_NAMES = ("q_codes", "k_codes", "v_codes", "do_codes", "v_half", "do_half", "q_codes_t", "do_codes_t", "v_codes_t",
            "q_scales", "k_scales", "v_scales", "do_scales", "l2", "drow", "dq_acc", "status")
TOK = 128  # token block of the INT8 operands; rows padded to a multiple of it
_lock = threading.Lock()
_declared = set()


def header_functions() -> list:
    """Names of the functions declared in include/sagebwd.h."""
    text = open(_HEADER).read()
    return sorted(set(re.findall(r"^[a-z_ 0-9\*]+?\b(sagebwd_[a-z_0-9]+)\s*\(", text, re.M)))


def lib() -> ctypes.CDLL:
    L = _fp4.load()
    with _lock:
        if id(L) not in _declared:
            vp, i, sz, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
            sig = {
                "sagebwd_workspace_bytes": (sz, [i, i, i, i]),
                "sagebwd_workspace_layout": (i, [i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]),
                "sagebwd_fwd": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]),
                "sagebwd_bwd": (i, [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]),
                "sagebwd_get_status": (i, [vp, i, i, i, i, vp]),
                "sagebwd_mma_peak": (i, [i, i, i, vp, vp]),
                "sagebwd_int_mma_probe": (i, [vp, vp, i, vp, vp]),
                "sagebwd_quantize_qkv": (i, [vp, vp, vp, i, i, i, i, vp, sz, vp]),
                "sagebwd_attn_fwd": (i, [vp, vp, i, i, i, i, i, f, vp, sz, vp]),
                "sagebwd_bwd_prep": (i, [vp, vp, vp, i, i, i, i, vp, sz, vp]),
                "sagebwd_attn_bwd": (i, [vp, vp, i, i, i, i, i, f, vp, sz, vp]),
                "sagebwd_dq_out": (i, [vp, i, i, i, i, vp, sz, vp]),
                "sagebwd_stall_test": (i, [i, vp, vp, i, i, i, i, f, ctypes.c_uint64, vp, sz, vp]),
                "sagebwd_umma_probe": (i, [vp, vp, i, vp, vp, vp]),
                "sagebwd_umma_mn_probe": (i, [vp, vp, vp, vp, vp]),
                "sagebwd_umma_ta_probe": (i, [vp, vp, i, vp, vp, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype, fn.argtypes = res, args
            _declared.add(id(L))
    return L


# ------------------------------------------------------------- raw entry points
def sagebwd_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return lib().sagebwd_workspace_bytes(B, H, N, D)


def sagebwd_workspace_layout(B: int, H: int, N: int, D: int):
    offs = (ctypes.c_size_t * WS_FIELDS)()
    rc = lib().sagebwd_workspace_layout(B, H, N, D, offs)
    return rc, list(offs)


def sagebwd_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, D, causal, scale, ws_ptr, ws_bytes,
                stream) -> int:
    return lib().sagebwd_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, D, int(causal), float(scale),
                             ws_ptr, ws_bytes, stream)


def sagebwd_bwd(do_ptr, o_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, B, H, N, D, causal, scale, ws_ptr,
                ws_bytes, stream) -> int:
    return lib().sagebwd_bwd(do_ptr, o_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, B, H, N, D, int(causal),
                             float(scale), ws_ptr, ws_bytes, stream)


def sagebwd_quantize_qkv(q_ptr, k_ptr, v_ptr, B, H, N, D, ws_ptr, ws_bytes, stream) -> int:
    return lib().sagebwd_quantize_qkv(q_ptr, k_ptr, v_ptr, B, H, N, D, ws_ptr, ws_bytes, stream)


def sagebwd_attn_fwd(o_ptr, lse_ptr, B, H, N, D, causal, scale, ws_ptr, ws_bytes, stream) -> int:
    return lib().sagebwd_attn_fwd(o_ptr, lse_ptr, B, H, N, D, int(causal), float(scale), ws_ptr, ws_bytes, stream)


def sagebwd_bwd_prep(do_ptr, o_ptr, lse_ptr, B, H, N, D, ws_ptr, ws_bytes, stream) -> int:
    return lib().sagebwd_bwd_prep(do_ptr, o_ptr, lse_ptr, B, H, N, D, ws_ptr, ws_bytes, stream)


def sagebwd_attn_bwd(dk_ptr, dv_ptr, B, H, N, D, causal, scale, ws_ptr, ws_bytes, stream) -> int:
    return lib().sagebwd_attn_bwd(dk_ptr, dv_ptr, B, H, N, D, int(causal), float(scale), ws_ptr, ws_bytes, stream)


def sagebwd_dq_out(dq_ptr, B, H, N, D, ws_ptr, ws_bytes, stream) -> int:
    return lib().sagebwd_dq_out(dq_ptr, B, H, N, D, ws_ptr, ws_bytes, stream)


def sagebwd_stall_test(kernel, out0_ptr, out1_ptr, B, H, N, D, scale, wait_limit_ns, ws_ptr, ws_bytes,
                       stream) -> int:
    return lib().sagebwd_stall_test(kernel, out0_ptr, out1_ptr, B, H, N, D, float(scale), wait_limit_ns, ws_ptr,
                                    ws_bytes, stream)


def sagebwd_get_status(ws_ptr, B, H, N, D, stream) -> int:
    return lib().sagebwd_get_status(ws_ptr, B, H, N, D, stream)


def sagebwd_mma_peak(kind: int, ctas: int, iters: int, scratch_ptr, stream) -> int:
    return lib().sagebwd_mma_peak(kind, ctas, iters, scratch_ptr, stream)


def sagebwd_umma_probe(a_ptr, b_ptr, N: int, c_ptr, status_ptr, stream) -> int:
    return lib().sagebwd_umma_probe(a_ptr, b_ptr, N, c_ptr, status_ptr, stream)


def sagebwd_umma_ta_probe(a_ptr, b_ptr, N: int, c_ptr, status_ptr, stream) -> int:
    return lib().sagebwd_umma_ta_probe(a_ptr, b_ptr, N, c_ptr, status_ptr, stream)


def sagebwd_umma_mn_probe(a_ptr, b_ptr, c_ptr, status_ptr, stream) -> int:
    return lib().sagebwd_umma_mn_probe(a_ptr, b_ptr, c_ptr, status_ptr, stream)


def sagebwd_int_mma_probe(a_ptr, b_ptr, K: int, out_ptr, stream) -> int:
    return lib().sagebwd_int_mma_probe(a_ptr, b_ptr, K, out_ptr, stream)


# ------------------------------------------------------------- torch conveniences
def default_scale(D: int) -> float:
    return D ** -0.5


class Workspace:
    """The device workspace one forward fills and its backward reads."""

    def __init__(self, B: int, H: int, N: int, D: int, device=None):
        import torch
        self.B, self.H, self.N, self.D = B, H, N, D
        self.nbytes = sagebwd_workspace_bytes(B, H, N, D)
        if self.nbytes == 0:
            raise SageFp4Error(EINVAL, f"SageBwd workspace for B={B} H={H} N={N} D={D}")
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        rc, self.offsets = sagebwd_workspace_layout(B, H, N, D)
        _fp4._check(rc, "sagebwd_workspace_layout")

    def fits(self, B, H, N, D) -> bool:
        return (self.B, self.H, self.N, self.D) == (B, H, N, D)

    def region(self, name: str):
        """Raw bytes of one region (for tests and inspection)."""
        i = WS_NAMES.index(name)
        end = self.offsets[i + 1] if i + 1 < WS_FIELDS else self.nbytes
        return self.buf[self.offsets[i]:end]

    def get_status(self, stream=None) -> int:
        return sagebwd_get_status(self.buf.data_ptr(), self.B, self.H, self.N, self.D, _fp4._stream(stream))


def _check_input(x, shape, name):
    import torch
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise SageFp4Error(EINVAL, f"{name} must be a contiguous bf16 CUDA tensor")
    if tuple(x.shape) != tuple(shape):
        raise SageFp4Error(EINVAL, f"{name} has shape {tuple(x.shape)}, expected {tuple(shape)}")


def forward(q, k, v, causal: bool = False, scale=None, workspace: Workspace | None = None, stream=None):
    """SageBwd forward on bf16 [B, H, N, D] tensors.  Returns (o, lse, workspace);
    the workspace carries the quantized Q, K, V to the backward."""
    import torch
    B, H, N, D = q.shape
    for x, nm in ((q, "q"), (k, "k"), (v, "v")):
        _check_input(x, (B, H, N, D), nm)
    scale = default_scale(D) if scale is None else float(scale)
    ws = workspace if workspace is not None and workspace.fits(B, H, N, D) else Workspace(B, H, N, D, q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _fp4._order_after_current(stream, q, k, v, o, lse, ws.buf)
    _fp4._check(sagebwd_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, D,
                            causal, scale, ws.buf.data_ptr(), ws.nbytes, _fp4._stream(stream)), "sagebwd_fwd")
    return o, lse, ws


def backward(dout, o, lse, workspace: Workspace, causal: bool = False, scale=None, stream=None):
    """SageBwd backward: dq, dk, dv (bf16) of the forward that filled `workspace`."""
    import torch
    B, H, N, D = o.shape
    _check_input(dout, (B, H, N, D), "dout")
    _check_input(o, (B, H, N, D), "o")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise SageFp4Error(EINVAL, "lse must be a contiguous float32 [B, H, N] tensor")
    if not workspace.fits(B, H, N, D):
        raise SageFp4Error(EINVAL, "the workspace belongs to another problem size")
    scale = default_scale(D) if scale is None else float(scale)
    dq, dk, dv = (torch.empty_like(o) for _ in range(3))
    _fp4._order_after_current(stream, dout, o, lse, dq, dk, dv, workspace.buf)
    _fp4._check(sagebwd_bwd(dout.data_ptr(), o.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                            dv.data_ptr(), B, H, N, D, causal, scale, workspace.buf.data_ptr(), workspace.nbytes,
                            _fp4._stream(stream)), "sagebwd_bwd")
    return dq, dk, dv


def _autograd_function():
    import torch

    class SageBwdAttention(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, causal, scale):
            o, lse, ws = forward(q, k, v, causal, scale)
            ctx.save_for_backward(o, lse)
            ctx.ws, ctx.causal, ctx.scale = ws, causal, scale
            return o

        @staticmethod
        def backward(ctx, dout):
            o, lse = ctx.saved_tensors
            dq, dk, dv = backward(dout.contiguous(), o, lse, ctx.ws, ctx.causal, ctx.scale)
            ctx.ws = None
            return dq, dk, dv, None, None

    return SageBwdAttention


_fn = None


def attention(q, k, v, causal: bool = False, scale=None):
    """Differentiable SageBwd attention on bf16 [B, H, N, D] tensors."""
    global _fn
    if _fn is None:
        _fn = _autograd_function()
    return _fn.apply(q, k, v, causal, default_scale(q.shape[-1]) if scale is None else float(scale))


def mma_peak_tops(kind: int, ctas: int | None = None, iters: int = 4096, repeats: int = 3) -> float:
    """Best of `repeats` timed probe launches, in TOP/s (INT8, kind 0) or
    TFLOP/s (FP16 with FP32 accumulation: kind 1 warp-level, kinds 2-4
    tcgen05 with N = 64, 128, 256, kind 5 N = 64 with A in tensor memory,
    kind 6 N = 64 with B MN-major)."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    ctas = ctas or (4 * sms if kind < 2 else sms)
    scratch = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    _fp4._check(sagebwd_mma_peak(kind, ctas, iters, scratch.data_ptr(), st.cuda_stream), "sagebwd_mma_peak")
    best = float("inf")
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        _fp4._check(sagebwd_mma_peak(kind, ctas, iters, scratch.data_ptr(), st.cuda_stream), "sagebwd_mma_peak")
        e1.record(st)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    if kind >= 2:
        if int(scratch.item()) != 0:
            raise SageFp4Error(int(scratch.item()), "sagebwd_mma_peak: tcgen05 completion wait ran out")
        n = (64, 128, 256, 64, 64)[kind - 2]
        return 2.0 * 128 * n * 16 * 8 * iters * ctas / (best * 1e-3) / 1e12
    macs = (16 * 8 * 32) if kind == 0 else (16 * 8 * 16)
    warps = 256 // 32
    return 2.0 * macs * 8 * iters * warps * ctas / (best * 1e-3) / 1e12
