"""Decode the SageBwd workspace's tiled INT8 / FP16 layouts back to plain
[BH, Np, D] arrays, for the bit-exact quantization tests.

The layout contract (include/sagebwd.h, csrc/sagebwd.cu):
* every tile is contiguous; a tile of R rows W bytes wide stores logical
  byte (r, b) at r*W + (((b >> 4) ^ sw(r)) << 4) + (b & 15), sw(r) being
  (r >> 1) & 3 for W = 64 and r & 7 otherwise;
* row tiles hold T tokens x D channels ([T][D], FP16 ones 2D bytes wide);
* transposed tiles hold D rows of T tokens, the tokens of each 32-token
  chunk in a fixed order: position k holds token pi32(k) (or rho32(k) for
  K's dQ copy).
This is byte bookkeeping only; no quantization arithmetic lives here.
"""
import numpy as np


def pi32(k):
    return (k & 16) | (((k >> 1) & 1) << 3) | (((k >> 2) & 3) << 1) | (k & 1)


def rho32(k):
    return (k & 16) | ((k >> 1) & 7) | ((k & 1) << 3)


def _swz_index(R, W):
    r = np.arange(R)[:, None]
    b = np.arange(W)[None, :]
    sw = ((r >> 1) & 3) if W == 64 else (r & 7)
    return r * W + (((b >> 4) ^ sw) << 4) + (b & 15)


def unswizzle(tiles: np.ndarray, R: int, W: int) -> np.ndarray:
    """tiles: uint8 [..., R*W] -> [..., R, W] logical bytes."""
    idx = _swz_index(R, W)
    return tiles[..., idx]


def decode_rows(region: np.ndarray, BH: int, Np: int, D: int, T: int) -> np.ndarray:
    """INT8 row tiles -> int8 [BH, Np, D]."""
    t = region[:BH * Np * D].reshape(BH, Np // T, T * D)
    return unswizzle(t, T, D).reshape(BH, Np, D).view(np.int8)


def decode_cols(region: np.ndarray, BH: int, Np: int, D: int, T: int, perm) -> np.ndarray:
    """INT8 transposed tiles -> int8 [BH, Np, D] in token order."""
    t = unswizzle(region[:BH * Np * D].reshape(BH, Np // T, T * D), D, T)  # [BH, tiles, D, T]
    p = np.arange(T)
    tok = (p & ~31) | perm(p & 31)
    out = np.empty((BH, Np // T, T, D), np.uint8)
    out[:, :, tok, :] = t.transpose(0, 1, 3, 2)
    return out.reshape(BH, Np, D).view(np.int8)


def decode_half(region: np.ndarray, BH: int, Np: int, D: int, T: int) -> np.ndarray:
    """FP16 row tiles -> float16 [BH, Np, D]."""
    t = region[:BH * Np * D * 2].reshape(BH, Np // T, T * 2 * D)
    return np.ascontiguousarray(unswizzle(t, T, 2 * D)).view(np.float16).reshape(BH, Np, D)
