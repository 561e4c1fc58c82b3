"""Test-side helpers: layout conversions and error metrics.

These restate the scale layout documented in include/sage_fp4.h in numpy
index arithmetic; they belong to neither the CUDA path nor the oracle.
"""
import numpy as np


def block_offsets(R: int, groups: int) -> np.ndarray:
    """Byte offset of (row r, group g) in the 128x4 block scale layout, as [R, groups]."""
    r = np.arange(R)[:, None]
    g = np.arange(groups)[None, :]
    return ((r // 128) * (groups // 4) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4


def block_to_plain(block: np.ndarray, R: int, groups: int) -> np.ndarray:
    """[.., R*groups] bytes in block layout -> [.., R, groups]."""
    off = block_offsets(R, groups)
    return block.reshape(*block.shape[:-1], R * groups)[..., off]


def plain_to_block(plain: np.ndarray) -> np.ndarray:
    """[.., R, groups] (R a multiple of 128, groups of 4) -> [.., R*groups] block layout."""
    R, groups = plain.shape[-2:]
    off = block_offsets(R, groups)
    out = np.zeros((*plain.shape[:-2], R * groups), np.uint8)
    out[..., off] = plain
    return out


def rel_l1(o: np.ndarray, ref: np.ndarray) -> float:
    return float(np.abs(o - ref).sum() / np.abs(ref).sum())


def cosine(o: np.ndarray, ref: np.ndarray) -> float:
    o = o.reshape(-1).astype(np.float64)
    ref = ref.reshape(-1).astype(np.float64)
    return float((o * ref).sum() / np.sqrt((o * o).sum() * (ref * ref).sum()))


def e2m1_table() -> np.ndarray:
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    return np.concatenate([mags, -mags])


def sample_rows(BH: int, N: int, per_head: int, seed: int = 0) -> np.ndarray:
    """Deterministic row sample: every (b,h); first and last row, first and last
    128-row tile's edges, and random rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for bh in range(BH):
        pick = {0, N - 1, min(127, N - 1), max(0, N - 128)}
        pick |= set(int(x) for x in rng.integers(0, N, size=max(0, per_head - len(pick))))
        rows.extend(bh * N + i for i in sorted(pick))
    return np.array(rows, np.int64)
