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


# Tolerances of the GPU attention output against the oracle.  The whole
# tensor: relative L1 <= 5e-3 and cosine >= 0.999 (the target's).  Each row on
# its own: cosine >= 0.9995, and max |got - ref| <= ROW_MAXABS_K * max |ref| of
# that row, so that one bad row (left unwritten, stale, or from the wrong tile)
# cannot hide in the whole-tensor figures.  The two sides differ by bf16
# rounding of O (2^-9 relative) and by P codes at an E2M1 rounding boundary,
# where the kernel's FP32 exp2 and the oracle's FP64 exp can pick neighbouring
# codes.  Measured over every attention test case on GB300 (NVFP4 and MXFP4,
# all shapes): the worst row has max |diff| = 0.0055 of its largest value and
# cosine 0.99999; the bounds leave a margin of about 3.6x and 50x.
REL_L1_MAX = 5e-3
COS_MIN = 0.999
ROW_COS_MIN = 0.9995
ROW_MAXABS_K = 0.02


def row_stats(got: np.ndarray, ref: np.ndarray):
    """Per-row cosine and max |got - ref| / max |ref| for [rows, D] arrays.
    A row whose reference is all zero counts as matching only if the output
    row is zero too."""
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    ng, nr = np.sqrt((g * g).sum(1)), np.sqrt((r * r).sum(1))
    zero = nr == 0
    cos = np.where(zero, np.where(ng == 0, 1.0, 0.0), (g * r).sum(1) / np.where(zero, 1.0, ng * nr))
    rmax = np.abs(r).max(1)
    err = np.where(zero, np.where(np.abs(g).max(1) == 0, 0.0, np.inf),
                   np.abs(g - r).max(1) / np.where(zero, 1.0, rmax))
    return cos, err


def check_o(got: np.ndarray, ref: np.ndarray, label: str = "") -> dict:
    """Assert the GPU output `got` matches the oracle `ref` ([rows, D]) on the
    whole tensor and row by row; return the figures."""
    assert np.isfinite(got).all(), f"{label}: non-finite output rows " \
        f"{np.unique(np.argwhere(~np.isfinite(got))[:, 0])[:8]}"
    e, c = rel_l1(got, ref), cosine(got, ref)
    rc, re = row_stats(got, ref)
    worst = int(np.argmax(re))
    out = {"rel_l1": e, "cos": c, "row_cos_min": float(rc.min()), "row_err_max": float(re.max()),
           "worst_row": worst}
    print(f"{label}: rel-L1 {e:.2e} cos {c:.6f}; rows: min cos {rc.min():.5f}, "
          f"max |d|/max|ref| {re.max():.4f} (row {worst})")
    assert e <= REL_L1_MAX and c >= COS_MIN, (label, e, c)
    bad = np.argwhere((rc < ROW_COS_MIN) | (re > ROW_MAXABS_K))[:, 0]
    assert bad.size == 0, (label, "rows", bad[:8], rc[bad[:8]], re[bad[:8]])
    return out
