"""CPU oracle for SageAttention3's microscaled FP4 attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library (``bit_attention_gb300``) never imports, links or calls it, and the two
share no code: this wrapper marshals numpy arrays into the plain C oracle in
``sage_oracle.c`` and nothing else.

The method follows the senqingzn.com article on SageAttention3 (sections
"Solving two obstacles and one difficulty" and "FP4 attention inference
acceleration and hardware implementation/optimisation") and the abstract of
"SageAttention3: Microscaling FP4 Attention for Inference and An Exploration
of 8-Bit Training".  See ``sage_oracle.c`` for the step-by-step definition.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "sage_oracle.c")
_SRC_BWD = os.path.join(_HERE, "sagebwd_oracle.c")  # SageBwd, the 8-bit attention for training
_lock = threading.Lock()
_lib = None

PMODE = {"tile": 0, "running": 1}
# normaliser l: from the unquantized probabilities (the method's reading), or
# from the rounded probabilities that enter PV (Direct-P)
LNORM = {"exp": 0, "rounded": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    srcs = [_SRC, _SRC_BWD]
    deps = srcs + [s[:-2] + ".h" for s in srcs]
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in deps)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", *srcs, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load(path: str):
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _load(_LIB_PATH)
    return _lib


class swapped:
    """Context manager: route this module's calls through another build of the
    oracle (used by the tests that plant mistakes in a copy of the source)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        lib()
        self.saved = _lib
        _lib = _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _declare(L):
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    L.sor_e2m1_value.restype = ctypes.c_double
    L.sor_e2m1_value.argtypes = [ctypes.c_int]
    L.sor_e2m1_encode.restype = ctypes.c_int
    L.sor_e2m1_encode.argtypes = [ctypes.c_float]
    L.sor_e4m3_value.restype = ctypes.c_double
    L.sor_e4m3_value.argtypes = [ctypes.c_int]
    L.sor_e4m3_encode.restype = ctypes.c_int
    L.sor_e4m3_encode.argtypes = [ctypes.c_float]
    L.sor_encode_range.restype = None
    L.sor_encode_range.argtypes = [ctypes.c_uint32, ctypes.c_uint32, u8p, u8p]
    L.sor_quant_group16.restype = None
    L.sor_quant_group16.argtypes = [f32p, u8p, u8p]
    L.sor_quantize_rows.restype = None
    L.sor_quantize_rows.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p, u8p]
    L.sor_quantize_v.restype = None
    L.sor_quantize_v.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p, u8p]
    L.sor_e8m0_value.restype = ctypes.c_double
    L.sor_e8m0_value.argtypes = [ctypes.c_int]
    L.sor_quant_group32_mx.restype = None
    L.sor_quant_group32_mx.argtypes = [f32p, u8p, u8p]
    for fn in (L.sor_quantize_rows_fmt, L.sor_quantize_v_fmt):
        fn.restype = None
        fn.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p, u8p]
    L.sor_attention_ex.restype = ctypes.c_int
    L.sor_attention_ex.argtypes = [u8p, u8p, u8p, u8p, u8p, u8p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int64,
                                   f64p, f64p, f64p]
    L.sor_attention.restype = ctypes.c_int
    L.sor_attention.argtypes = [u8p, u8p, u8p, u8p, u8p, u8p, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int64, f64p, f64p, f64p]
    # SageBwd (absent from the one-file builds the mutation tests make)
    if hasattr(L, "sbo_attention_train"):
        L.sbo_int8_code.restype = ctypes.c_int
        L.sbo_int8_code.argtypes = [ctypes.c_float, ctypes.c_float]
        L.sbo_int8_scale.restype = ctypes.c_float
        L.sbo_int8_scale.argtypes = [ctypes.c_float]
        L.sbo_quantize_blocks.restype = None
        L.sbo_quantize_blocks.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int8), f32p]
        L.sbo_attention_train.restype = ctypes.c_int
        L.sbo_attention_train.argtypes = [u16p, u16p, u16p, u16p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                          f64p, f64p, f64p, f64p, f64p]
    L.sor_attention_exact.restype = ctypes.c_int
    L.sor_attention_exact.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_double, i64p,
                                      ctypes.c_int64, f64p]
    L.sor_num_threads.restype = ctypes.c_int


def _p(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(x) -> np.ndarray:
    """bf16 data as its raw 16-bit patterns (accepts torch bf16 tensors or uint16 arrays)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


# ---------------------------------------------------------------- codecs
def e2m1_value(code: int) -> float:
    return lib().sor_e2m1_value(int(code))


def e2m1_encode(x: float) -> int:
    return lib().sor_e2m1_encode(float(x))


def e4m3_value(bits: int) -> float:
    return lib().sor_e4m3_value(int(bits))


def e4m3_encode(x: float) -> int:
    return lib().sor_e4m3_encode(float(x))


def encode_range(first: int, count: int):
    e2 = np.empty(count, np.uint8)
    e4 = np.empty(count, np.uint8)
    lib().sor_encode_range(first, count, _p(e2, ctypes.c_uint8), _p(e4, ctypes.c_uint8))
    return e2, e4


def e8m0_value(bits: int) -> float:
    return lib().sor_e8m0_value(int(bits))


def quant_group32_mx(x):
    """MXFP4 group: 32 floats -> (32 E2M1 codes, E8M0 scale byte)."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    assert x.shape == (32,)
    codes = np.empty(32, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().sor_quant_group32_mx(_p(x, ctypes.c_float), _p(codes, ctypes.c_uint8), _p(sc, ctypes.c_uint8))
    return codes, int(sc[0])


def quant_group16(x):
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    assert x.shape == (16,)
    codes = np.empty(16, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().sor_quant_group16(_p(x, ctypes.c_float), _p(codes, ctypes.c_uint8), _p(sc, ctypes.c_uint8))
    return codes, int(sc[0])


# ------------------------------------------------------------ quantizers
FORMATS = {"nvfp4": 0, "mxfp4": 1}   # microscaling format -> oracle code
GROUP = {"nvfp4": 16, "mxfp4": 32}   # elements per scale


def quantize_rows(x, BH: int, N: int, D: int, fmt: str = "nvfp4"):
    """Q/K: bf16 [BH,N,D] -> codes [BH,N_pad,D/2], scales [BH,N_pad,D/G] (plain layout)."""
    x = _u16(x).reshape(-1)
    assert x.size == BH * N * D
    Np = round_up(N, 128)
    codes = np.empty((BH, Np, D // 2), np.uint8)
    scales = np.empty((BH, Np, D // GROUP[fmt]), np.uint8)
    lib().sor_quantize_rows_fmt(_p(x, ctypes.c_uint16), BH, N, D, FORMATS[fmt],
                                _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8))
    return codes, scales


def quantize_v(v, BH: int, N: int, D: int, fmt: str = "nvfp4"):
    """V: bf16 [BH,N,D] -> V^T codes [BH,D,N_pad/2], scales [BH,D,N_pad/G] (plain layout)."""
    v = _u16(v).reshape(-1)
    assert v.size == BH * N * D
    Np = round_up(N, 128)
    codes = np.empty((BH, D, Np // 2), np.uint8)
    scales = np.empty((BH, D, Np // GROUP[fmt]), np.uint8)
    lib().sor_quantize_v_fmt(_p(v, ctypes.c_uint16), BH, N, D, FORMATS[fmt],
                             _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8))
    return codes, scales


class Quantized:
    """The oracle's quantized Q, K, V^T for one problem, in one microscaling format."""

    def __init__(self, q, k, v, BH: int, N: int, D: int, fmt: str = "nvfp4"):
        self.BH, self.N, self.D, self.fmt = BH, N, D, fmt
        self.qc, self.qs = quantize_rows(q, BH, N, D, fmt)
        self.kc, self.ks = quantize_rows(k, BH, N, D, fmt)
        self.vc, self.vs = quantize_v(v, BH, N, D, fmt)


# ------------------------------------------------------------- attention
def default_scale(D: int) -> float:
    """Softmax scale when none is given: 1/sqrt(D) (the pages name none)."""
    return 1.0 / math.sqrt(D)


def attention(qz: Quantized, causal: bool, pmode: str = "tile", rows=None, kv_tile: int = 128,
              scale: float | None = None, lnorm: str = "exp"):
    """Tiled FP4 attention. Returns (O [nrows,D] float64, l [nrows], m [nrows]).
    lnorm: "exp" (l from the unquantized probabilities) or "rounded" (Direct-P)."""
    BH, N, D = qz.BH, qz.N, qz.D
    scale = default_scale(D) if scale is None else float(scale)
    if rows is None:
        rows_a = None
        nrows = BH * N
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, np.int64))
        nrows = rows_a.size
    out = np.empty((nrows, D), np.float64)
    ol = np.empty(nrows, np.float64)
    om = np.empty(nrows, np.float64)
    rc = lib().sor_attention_ex(
        _p(qz.qc, ctypes.c_uint8), _p(qz.qs, ctypes.c_uint8), _p(qz.kc, ctypes.c_uint8),
        _p(qz.ks, ctypes.c_uint8), _p(qz.vc, ctypes.c_uint8), _p(qz.vs, ctypes.c_uint8),
        BH, N, D, int(bool(causal)), FORMATS[qz.fmt], scale, PMODE[pmode], LNORM[lnorm], kv_tile,
        _p(rows_a, ctypes.c_int64) if rows_a is not None else None, nrows,
        _p(out, ctypes.c_double), _p(ol, ctypes.c_double), _p(om, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle attention rejected its arguments")
    return out, ol, om


def attention_exact(q, k, v, BH: int, N: int, D: int, causal: bool, rows=None,
                    scale: float | None = None):
    """Unquantized softmax(scale QK^T)V in float64 from the bf16 inputs (scale 1/sqrt(D))."""
    scale = default_scale(D) if scale is None else float(scale)
    q, k, v = _u16(q).reshape(-1), _u16(k).reshape(-1), _u16(v).reshape(-1)
    if rows is None:
        rows_a, nrows = None, BH * N
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, np.int64))
        nrows = rows_a.size
    out = np.empty((nrows, D), np.float64)
    rc = lib().sor_attention_exact(
        _p(q, ctypes.c_uint16), _p(k, ctypes.c_uint16), _p(v, ctypes.c_uint16), BH, N, D,
        int(bool(causal)), scale, _p(rows_a, ctypes.c_int64) if rows_a is not None else None, nrows,
        _p(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle exact attention rejected its arguments")
    return out


def num_threads() -> int:
    return lib().sor_num_threads()


# -------------------------------------------------- decoding helpers
def decode_rows(codes: np.ndarray, scales: np.ndarray, fmt: str = "nvfp4") -> np.ndarray:
    """Decode [.., R, C/2] codes and [.., R, C/G] scales (plain layout) to float64 [.., R, C]."""
    e2 = np.array([e2m1_value(i) for i in range(16)])
    dec = e4m3_value if fmt == "nvfp4" else e8m0_value
    sv = np.array([dec(i) for i in range(256)])
    lo = codes & 0x0F
    hi = codes >> 4
    el = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    vals = e2[el]
    sc = np.repeat(sv[scales], GROUP[fmt], axis=-1)
    return vals * sc


# ------------------------------------------------------------------ SageBwd
SAGEBWD_BLOCK = 128  # token block of the INT8 operands Q, K, V, dO; key edge of a P / dS block
SAGEBWD_QBLOCK = 64  # query edge of a P / dS block


def int8_code(x: float, amax: float) -> int:
    return lib().sbo_int8_code(x, amax)


def int8_scale(amax: float) -> float:
    return lib().sbo_int8_scale(amax)


def sagebwd_quantize(x, BH: int, N: int, D: int):
    """bf16 [.., N, D] -> (INT8 codes [BH, N, D], float scales [BH, ceil(N/128)])."""
    xb = _u16(x)
    nb = (N + SAGEBWD_BLOCK - 1) // SAGEBWD_BLOCK
    codes = np.empty((BH, N, D), np.int8)
    scales = np.empty((BH, nb), np.float32)
    lib().sbo_quantize_blocks(_p(xb, ctypes.c_uint16), BH, N, D, _p(codes, ctypes.c_int8),
                              _p(scales, ctypes.c_float))
    return codes, scales


def sagebwd(q, k, v, dout, BH: int, N: int, D: int, causal: bool, scale: float | None = None,
            quant: bool = True):
    """SageBwd forward and backward. Returns (o, lse, dq, dk, dv), float64,
    [BH, N, D] (lse [BH, N]).  quant=False: exact attention and its gradient."""
    scale = default_scale(D) if scale is None else float(scale)
    bufs = [_u16(t) for t in (q, k, v, dout)]
    o = np.empty((BH, N, D), np.float64)
    lse = np.empty((BH, N), np.float64)
    dq, dk, dv = (np.empty((BH, N, D), np.float64) for _ in range(3))
    rc = lib().sbo_attention_train(*(_p(b, ctypes.c_uint16) for b in bufs), BH, N, D, int(bool(causal)),
                                   scale, int(bool(quant)), *(_p(a, ctypes.c_double) for a in (o, lse, dq, dk, dv)))
    if rc != 0:
        raise ValueError(f"SageBwd oracle failed ({rc})")
    return o, lse, dq, dk, dv
