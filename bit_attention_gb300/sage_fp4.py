"""Thin Python binding of the C ABI in ``include/sage_fp4.h``.

Argument marshalling only: every step of the attention path runs in the CUDA
kernels of ``_build/libsagefp4.so``.  PyTorch provides device memory and
streams.  There is no fallback: if the library cannot be built or loaded, or a
call fails, an exception is raised.

Functions named ``sage_fp4_*`` mirror the C entry points one to one and take
raw device pointers; ``quantize_qkv`` and ``attn_fwd`` are the torch-tensor
conveniences built on them.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re
import threading

from . import build as _build

OK, EINVAL, ECUDA, ETIMEOUT, EUNSUPPORTED, ETOOLARGE, EBOUNDS = 0, -1, -2, -3, -4, -5, -6
# SAGE_FP4_FORMAT_*; "mxfp4_directp": MXFP4 with the softmax normaliser summed
# from the rounded P (Direct-P); its operands are MXFP4
FORMATS = {"nvfp4": 0, "mxfp4": 1, "mxfp4_directp": 2}

_HEADER = os.path.join(_build.ROOT, "include", "sage_fp4.h")
_lock = threading.Lock()
_libs = {}             # loaded libraries: False = release, True = bounds-checking debug build
_use_debug = False     # which one the calls below go to (debug_bounds_library())


class SageFp4Error(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (status {code})")
        self.code = code


class sage_fp4_tensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class sage_fp4_strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("n", ctypes.c_int64)]


class sage_fp4_qkv(ctypes.Structure):
    _fields_ = [("q", sage_fp4_tensor), ("k", sage_fp4_tensor), ("vt", sage_fp4_tensor),
                ("status", ctypes.c_void_p)]


def header_functions() -> list:
    """Names of the functions declared in include/sage_fp4.h."""
    text = open(_HEADER).read()
    return sorted(set(re.findall(r"^[a-z_ 0-9\*]+?\b(sage_fp4_[a-z_0-9]+)\s*\(", text, re.M)))


def load(build: bool = True, debug_bounds: bool | None = None) -> ctypes.CDLL:
    """Load the library, building it first when it is missing or stale.

    debug_bounds: the build whose kernels check every computed index against
    its buffer (SAGE_FP4_EBOUNDS); None = the one debug_bounds_library()
    selects (the release library outside it)."""
    dbg = _use_debug if debug_bounds is None else bool(debug_bounds)
    with _lock:
        if dbg not in _libs:
            path = _build.build(debug_bounds=dbg) if build else (_build.LIB_DEBUG if dbg else _build.LIB)
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path}")
            L = ctypes.CDLL(path)
            vp, i, sz, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint32
            qp = ctypes.POINTER(sage_fp4_qkv)
            sp = ctypes.POINTER(sage_fp4_strides)
            sig = {
                "sage_fp4_workspace_bytes": (sz, [i, i, i, i]),
                "sage_fp4_qkv_from_workspace": (i, [vp, sz, i, i, i, i, qp]),
                "sage_fp4_quantize_qkv": (i, [vp, vp, vp, qp, i, i, i, i, vp]),
                "sage_fp4_attn_fwd": (i, [qp, vp, i, i, i, i, i, vp]),
                "sage_fp4_quantize_qkv_strided": (i, [vp, sp, vp, sp, vp, sp, qp, i, i, i, i, i, vp]),
                "sage_fp4_attn_fwd_ex": (i, [qp, vp, sp, i, i, i, i, i, ctypes.c_float, i, vp]),
                "sage_fp4_attn_fwd_stall_test": (i, [qp, vp, i, i, i, i, i, ctypes.c_uint64, vp]),
                "sage_fp4_quantize_qkv_stall_test": (i, [vp, vp, vp, qp, i, i, i, i, ctypes.c_uint64, vp]),
                "sage_fp4_get_status": (i, [qp, vp]),
                "sage_fp4_strerror": (ctypes.c_char_p, [i]),
                "sage_fp4_cvt_probe": (i, [u32, u32, vp, vp, vp]),
                "sage_fp4_mma_probe": (i, [vp, vp, vp, vp, i, i, i, vp, vp, vp]),
                "sage_fp4_mma_probe_mx": (i, [vp, vp, vp, vp, i, i, i, vp, vp, vp]),
                "sage_fp4_mma_probe_ex": (i, [vp, vp, vp, vp, i, i, i, vp, vp, vp]),
                "sage_fp4_mma_peak": (i, [i, i, vp, vp]),
                "sage_fp4_tmem_max_probe": (i, [vp, vp, vp, vp]),
                "sage_fp4_attention_noalloc": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, vp]),
                "sage_fp4_host_workspace_bytes": (sz, [i, i, i, i]),
                "sage_fp4_attention_host": (i, [vp, vp, vp, vp, i, i, i, i, i, vp, sz, vp, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype, fn.argtypes = res, args
            _libs[dbg] = L
    return _libs[dbg]


@contextlib.contextmanager
def debug_bounds_library():
    """Route every call of this module to the bounds-checking debug build of
    the library while the block runs (for tests; not thread-safe)."""
    global _use_debug
    prev = _use_debug
    _use_debug = True
    try:
        yield load()
    finally:
        _use_debug = prev


def strerror(code: int) -> str:
    try:
        return load().sage_fp4_strerror(int(code)).decode()
    except Exception:  # the library itself failed to load
        return f"status {code}"


def _check(code: int, what: str) -> int:
    if code != OK:
        raise SageFp4Error(code, what)
    return code


# ------------------------------------------------------------- raw entry points
def sage_fp4_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return load().sage_fp4_workspace_bytes(B, H, N, D)


def sage_fp4_qkv_from_workspace(ws_ptr: int, ws_bytes: int, B: int, H: int, N: int, D: int):
    out = sage_fp4_qkv()
    rc = load().sage_fp4_qkv_from_workspace(ws_ptr, ws_bytes, B, H, N, D, ctypes.byref(out))
    return rc, out


def sage_fp4_quantize_qkv(q_ptr, k_ptr, v_ptr, qkv: sage_fp4_qkv, B, H, N, D, stream) -> int:
    return load().sage_fp4_quantize_qkv(q_ptr, k_ptr, v_ptr, ctypes.byref(qkv), B, H, N, D, stream)


def sage_fp4_attn_fwd(qkv: sage_fp4_qkv, o_ptr, B, H, N, D, causal, stream) -> int:
    return load().sage_fp4_attn_fwd(ctypes.byref(qkv), o_ptr, B, H, N, D, int(causal), stream)


def sage_fp4_quantize_qkv_strided(q_ptr, q_strides, k_ptr, k_strides, v_ptr, v_strides,
                                  qkv: sage_fp4_qkv, B, H, N, D, stream, fmt: int = 0) -> int:
    """Strides: sage_fp4_strides or None (contiguous [B,H,N,D]); fmt: SAGE_FP4_FORMAT_*."""
    r = ctypes.byref
    return load().sage_fp4_quantize_qkv_strided(
        q_ptr, r(q_strides) if q_strides is not None else None, k_ptr,
        r(k_strides) if k_strides is not None else None, v_ptr,
        r(v_strides) if v_strides is not None else None, ctypes.byref(qkv), B, H, N, D, int(fmt),
        stream)


def sage_fp4_attn_fwd_ex(qkv: sage_fp4_qkv, o_ptr, o_strides, B, H, N, D, causal, softmax_scale,
                         stream, fmt: int = 0) -> int:
    return load().sage_fp4_attn_fwd_ex(ctypes.byref(qkv), o_ptr,
                                       ctypes.byref(o_strides) if o_strides is not None else None,
                                       B, H, N, D, int(causal), float(softmax_scale), int(fmt), stream)


def sage_fp4_attn_fwd_stall_test(qkv: sage_fp4_qkv, o_ptr, B, H, N, D, causal, wait_limit_ns,
                                 stream) -> int:
    return load().sage_fp4_attn_fwd_stall_test(ctypes.byref(qkv), o_ptr, B, H, N, D, int(causal),
                                               int(wait_limit_ns), stream)


def sage_fp4_quantize_qkv_stall_test(q_ptr, k_ptr, v_ptr, qkv: sage_fp4_qkv, B, H, N, D, wait_limit_ns,
                                     stream) -> int:
    return load().sage_fp4_quantize_qkv_stall_test(q_ptr, k_ptr, v_ptr, ctypes.byref(qkv), B, H, N, D,
                                                   int(wait_limit_ns), stream)


def sage_fp4_get_status(qkv: sage_fp4_qkv, stream) -> int:
    return load().sage_fp4_get_status(ctypes.byref(qkv), stream)


def sage_fp4_strerror(code: int) -> str:
    return strerror(code)


def sage_fp4_cvt_probe(first: int, count: int, e2m1_ptr, e4m3_ptr, stream) -> int:
    return load().sage_fp4_cvt_probe(first, count, e2m1_ptr, e4m3_ptr, stream)


def sage_fp4_mma_probe(a_codes, a_scales, b_codes, b_scales, n, K, a_by_threads, d, status,
                       stream) -> int:
    return load().sage_fp4_mma_probe(a_codes, a_scales, b_codes, b_scales, n, K,
                                     int(a_by_threads), d, status, stream)


def sage_fp4_mma_probe_mx(a_codes, a_scales, b_codes, b_scales, n, K, a_by_threads, d, status,
                          stream) -> int:
    return load().sage_fp4_mma_probe_mx(a_codes, a_scales, b_codes, b_scales, n, K, a_by_threads, d,
                                        status, stream)


PROBE_A_BY_THREADS, PROBE_MX, PROBE_SF_ROWS128 = 1, 2, 4


def sage_fp4_mma_probe_ex(a_codes, a_scales, b_codes, b_scales, n, K, flags, d, status,
                          stream) -> int:
    return load().sage_fp4_mma_probe_ex(a_codes, a_scales, b_codes, b_scales, n, K, int(flags), d,
                                        status, stream)


def sage_fp4_mma_peak(iters, n, status_ptr, stream) -> int:
    return load().sage_fp4_mma_peak(iters, n, status_ptr, stream)


def sage_fp4_tmem_max_probe(in_ptr, vals_ptr, maxes_ptr, stream) -> int:
    return load().sage_fp4_tmem_max_probe(in_ptr, vals_ptr, maxes_ptr, stream)


def mma_peak_tflops(n: int = 256, iters: int = 20000, repeats: int = 3) -> float:
    """Best of `repeats` timed launches of sage_fp4_mma_peak, in TFLOP/s."""
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    _check(sage_fp4_mma_peak(iters, n, status.data_ptr(), st.cuda_stream), "sage_fp4_mma_peak")
    best = float("inf")
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        _check(sage_fp4_mma_peak(iters, n, status.data_ptr(), st.cuda_stream), "sage_fp4_mma_peak")
        e1.record(st)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    if int(status.item()) != 0:
        raise SageFp4Error(int(status.item()), "sage_fp4_mma_peak")
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return 2.0 * 128 * n * 64 * iters * sms / (best * 1e-3) / 1e12


def sage_fp4_attention_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, status_ptr, B, H, N, D, causal,
                               stream) -> int:
    """One-call quantize + attention that allocates nothing (fixed device scratch)."""
    return load().sage_fp4_attention_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, status_ptr, B, H, N, D,
                                             int(causal), stream)


def sage_fp4_host_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return load().sage_fp4_host_workspace_bytes(B, H, N, D)


def sage_fp4_attention_host(q_ptr, k_ptr, v_ptr, o_ptr, B, H, N, D, causal, ws_ptr, ws_bytes,
                            status_ptr, stream) -> int:
    return load().sage_fp4_attention_host(q_ptr, k_ptr, v_ptr, o_ptr, B, H, N, D, int(causal),
                                          ws_ptr, ws_bytes, status_ptr, stream)


# ------------------------------------------------------------- torch conveniences
def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _order_after_current(stream, *tensors):
    """Work queued on `stream` follows the current stream's (where the tensors
    were allocated and zeroed), and the allocator keeps the tensors' memory
    until `stream` is done with it."""
    import torch
    if stream is None or stream == torch.cuda.current_stream():
        return
    stream.wait_stream(torch.cuda.current_stream())
    for t in tensors:
        t.record_stream(stream)


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


class QuantizedQKV:
    """NVFP4 Q, K, V^T in one workspace tensor, with torch views of each part."""

    def __init__(self, B: int, H: int, N: int, D: int, device=None):
        import torch
        self.B, self.H, self.N, self.D = B, H, N, D
        self.Np = _round_up(N, 128)
        nbytes = sage_fp4_workspace_bytes(B, H, N, D)
        if nbytes == 0:
            raise SageFp4Error(EINVAL, f"workspace for B={B} H={H} N={N} D={D}")
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")
        rc, self.struct = sage_fp4_qkv_from_workspace(self.workspace.data_ptr(), nbytes, B, H, N, D)
        _check(rc, "sage_fp4_qkv_from_workspace")

    def _view(self, ptr: int, shape):
        off = ptr - self.workspace.data_ptr()
        n = 1
        for s in shape:
            n *= s
        return self.workspace[off:off + n].view(*shape)

    @property
    def q_codes(self):
        return self._view(self.struct.q.codes, (self.B * self.H, self.Np, self.D // 2))

    @property
    def q_scales(self):
        return self._view(self.struct.q.scales, (self.B * self.H, self.Np * self.D // 16))

    @property
    def k_codes(self):
        return self._view(self.struct.k.codes, (self.B * self.H, self.Np, self.D // 2))

    @property
    def k_scales(self):
        return self._view(self.struct.k.scales, (self.B * self.H, self.Np * self.D // 16))

    @property
    def vt_codes(self):
        return self._view(self.struct.vt.codes, (self.B * self.H, self.D, self.Np // 2))

    @property
    def vt_scales(self):
        return self._view(self.struct.vt.scales, (self.B * self.H, 8 * self.Np))

    @property
    def status(self):
        return self._view(self.struct.status, (4,)).view(torch_int32())

    def get_status(self, stream=None) -> int:
        return sage_fp4_get_status(self.struct, _stream(stream))


def torch_int32():
    import torch
    return torch.int32


def _check_input(x, B, H, N, D, name):
    import torch
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise SageFp4Error(EINVAL, f"{name} must be a contiguous bf16 CUDA tensor")
    if tuple(x.shape) != (B, H, N, D):
        raise SageFp4Error(EINVAL, f"{name} has shape {tuple(x.shape)}, expected {(B, H, N, D)}")


def quantize_qkv(q, k, v, out: QuantizedQKV | None = None, stream=None,
                 fmt: str = "nvfp4") -> QuantizedQKV:
    """bf16 [B,H,N,D] Q, K, V on the GPU -> NVFP4 (or MXFP4) operands (one call, two kernels)."""
    B, H, N, D = q.shape
    for x, nm in ((q, "q"), (k, "k"), (v, "v")):
        _check_input(x, B, H, N, D, nm)
    if out is None:
        out = QuantizedQKV(B, H, N, D, device=q.device)
        _order_after_current(stream, out.workspace)
    if fmt == "nvfp4":
        rc = sage_fp4_quantize_qkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.struct, B, H, N, D,
                                   _stream(stream))
    else:
        rc = sage_fp4_quantize_qkv_strided(q.data_ptr(), None, k.data_ptr(), None, v.data_ptr(), None,
                                           out.struct, B, H, N, D, _stream(stream), _fmt(fmt))
    _check(rc, "sage_fp4_quantize_qkv")
    out.fmt = fmt
    return out


def _fmt(fmt: str) -> int:
    if fmt not in FORMATS:
        raise SageFp4Error(EINVAL, f"format must be one of {tuple(FORMATS)}, not {fmt!r}")
    return FORMATS[fmt]


def attn_fwd(qkv: QuantizedQKV, causal: bool = False, out=None, stream=None, scale=None):
    """SageAttention3 FP4 attention forward over quantized operands -> bf16 [B,H,N,D].

    scale: softmax scale (default 1/sqrt(D))."""
    import torch
    B, H, N, D = qkv.B, qkv.H, qkv.N, qkv.D
    if out is None:
        out = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=qkv.workspace.device)
    else:
        _check_input(out, B, H, N, D, "out")
    fmt = getattr(qkv, "fmt", "nvfp4")
    if scale is None and fmt == "nvfp4":
        rc = sage_fp4_attn_fwd(qkv.struct, out.data_ptr(), B, H, N, D, causal, _stream(stream))
    else:
        sc = 1.0 / (D ** 0.5) if scale is None else float(scale)
        rc = sage_fp4_attn_fwd_ex(qkv.struct, out.data_ptr(), None, B, H, N, D, causal, sc,
                                  _stream(stream), _fmt(fmt))
    _check(rc, "sage_fp4_attn_fwd")
    return out


LAYOUTS = ("HND", "NHD")


def _bhnd(x, layout: str, name: str):
    """(B, H, N, D) and the element strides of a bf16 CUDA tensor in `layout`
    (HND = [B,H,N,D], NHD = [B,N,H,D]); any strides with a contiguous D axis."""
    import torch
    if layout not in LAYOUTS:
        raise SageFp4Error(EINVAL, f"layout must be one of {LAYOUTS}, not {layout!r}")
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 4 or x.stride(3) != 1:
        raise SageFp4Error(EINVAL, f"{name} must be a 4-D bf16 CUDA tensor with a contiguous last axis")
    if layout == "HND":
        (B, H, N, D), (sb, sh, sn) = x.shape, x.stride()[:3]
    else:
        (B, N, H, D), (sb, sn, sh) = x.shape, x.stride()[:3]
    return (B, H, N, D), sage_fp4_strides(sb, sh, sn)


def attention(q, k, v, causal: bool = False, scale=None, layout: str = "HND", out=None,
              stream=None, fmt: str = "nvfp4"):
    """Plug-and-play SageAttention3 FP4 attention: bf16 Q, K, V -> bf16 O.

    layout: "HND" ([B,H,N,D]) or "NHD" ([B,N,H,D]); the tensors may be any
    views whose last axis is contiguous (e.g. slices of a packed QKV tensor),
    with 16-byte aligned rows.  scale: softmax scale (default 1/sqrt(D)).
    fmt: "nvfp4" (the method's) or "mxfp4" (the alternative the pages weighed).
    O is a new contiguous tensor in `layout` unless `out` is given.
    Quantization runs in a temporary workspace; three kernel launches."""
    import torch
    shape, sq = _bhnd(q, layout, "q")
    B, H, N, D = shape
    for x, nm in ((k, "k"), (v, "v")):
        if _bhnd(x, layout, nm)[0] != shape:
            raise SageFp4Error(EINVAL, f"{nm} has shape {tuple(x.shape)}, q has {tuple(q.shape)}")
    sk, sv = _bhnd(k, layout, "k")[1], _bhnd(v, layout, "v")[1]
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    elif _bhnd(out, layout, "out")[0] != shape:
        raise SageFp4Error(EINVAL, f"out has shape {tuple(out.shape)}, q has {tuple(q.shape)}")
    so = _bhnd(out, layout, "out")[1]
    z = QuantizedQKV(B, H, N, D, device=q.device)
    _order_after_current(stream, z.workspace, out)
    st = _stream(stream)
    f = _fmt(fmt)
    _check(sage_fp4_quantize_qkv_strided(q.data_ptr(), sq, k.data_ptr(), sk, v.data_ptr(), sv, z.struct,
                                         B, H, N, D, st, f), "sage_fp4_quantize_qkv_strided")
    sc = 1.0 / (D ** 0.5) if scale is None else float(scale)
    _check(sage_fp4_attn_fwd_ex(z.struct, out.data_ptr(), so, B, H, N, D, causal, sc, st, f),
           "sage_fp4_attn_fwd_ex")
    return out


class HostWorkspace:
    """Device workspace and status word of ``attention_host`` for one problem size."""

    def __init__(self, B: int, H: int, N: int, D: int, device=None):
        import torch
        self.B, self.H, self.N, self.D = B, H, N, D
        self.nbytes = sage_fp4_host_workspace_bytes(B, H, N, D)
        if self.nbytes == 0:
            raise SageFp4Error(EINVAL, f"host workspace for B={B} H={H} N={N} D={D}")
        dev = device or "cuda"
        self.workspace = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)

    def get_status(self, stream=None) -> int:
        """Synchronise, return the status word and reset it to 0."""
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        s.synchronize()
        v = int(self.status[0].item())
        self.status.zero_()
        return v


def _check_host(x, B, H, N, D, name):
    import torch
    if x.dtype != torch.bfloat16 or x.is_cuda or not x.is_contiguous():
        raise SageFp4Error(EINVAL, f"{name} must be a contiguous bf16 CPU tensor")
    if tuple(x.shape) != (B, H, N, D):
        raise SageFp4Error(EINVAL, f"{name} has shape {tuple(x.shape)}, expected {(B, H, N, D)}")


def attention_host(q, k, v, causal: bool = False, out=None, workspace: HostWorkspace | None = None,
                   stream=None):
    """Quantize and attend with Q, K, V and O in host memory (pin them for overlap).

    Asynchronous on ``stream`` like the device calls: synchronise it before
    reading ``out``."""
    import torch
    B, H, N, D = q.shape
    for x, nm in ((q, "q"), (k, "k"), (v, "v")):
        _check_host(x, B, H, N, D, nm)
    if out is None:
        out = torch.empty((B, H, N, D), dtype=torch.bfloat16, pin_memory=True)
    else:
        _check_host(out, B, H, N, D, "out")
    if workspace is None:
        workspace = HostWorkspace(B, H, N, D)
    rc = sage_fp4_attention_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N,
                                 D, causal, workspace.workspace.data_ptr(), workspace.nbytes,
                                 workspace.status.data_ptr(), _stream(stream))
    _check(rc, "sage_fp4_attention_host")
    return out
