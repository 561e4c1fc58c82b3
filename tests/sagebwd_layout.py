"""Decode the SageBwd workspace's operand arrays back to plain [BH, Np, D]
arrays, for the bit-exact quantization tests.

The layout contract (include/sagebwd.h, csrc/sagebwd.cu): every operand is
FP16 rows [BH][Np][D] (2D bytes each) whose 16-byte chunks are XOR-permuted
by the row index: logical byte b of row r sits at
r*2D + (((b >> 4) ^ (r & 7)) << 4) + (b & 15).  INT8 codes are held as FP16
values.  This is byte bookkeeping only; no quantization arithmetic lives here.
"""
import numpy as np


def _swz_index(R, W):
    r = np.arange(R)[:, None]
    b = np.arange(W)[None, :]
    return r * W + (((b >> 4) ^ (r & 7)) << 4) + (b & 15)


def decode_half(region: np.ndarray, BH: int, Np: int, D: int) -> np.ndarray:
    """uint8 region -> float16 [BH, Np, D] in logical order."""
    rows = region[:BH * Np * 2 * D].reshape(BH, Np * 2 * D)
    return np.ascontiguousarray(rows[:, _swz_index(Np, 2 * D)]).view(np.float16).reshape(BH, Np, D)


def decode_codes(region: np.ndarray, BH: int, Np: int, D: int) -> np.ndarray:
    """INT8 codes held as FP16 values -> int8 [BH, Np, D]; every value must
    be an integer in [-127, 127]."""
    h = decode_half(region, BH, Np, D).astype(np.float64)
    assert np.all(h == np.rint(h)) and np.abs(h).max() <= 127
    return h.astype(np.int8)


def decode_codes_t(region: np.ndarray, BH: int, Np: int, D: int) -> np.ndarray:
    """Transposed code tiles ([64-token tile][D][64], rows of 128 bytes,
    swizzled) -> int8 [BH, Np, D] in token order."""
    t = region[:BH * Np * D * 2].reshape(BH, Np // 64, D * 128)
    h = np.ascontiguousarray(t[:, :, _swz_index(D, 128)]).view(np.float16).reshape(BH, Np // 64, D, 64)
    h = h.astype(np.float64)
    assert np.all(h == np.rint(h)) and np.abs(h).max() <= 127
    return h.transpose(0, 1, 3, 2).reshape(BH, Np, D).astype(np.int8)
