"""Pins for the oracle's codecs and its 1x16 group quantizer.

Each check compares the oracle with something other than itself: facts the
pages state (tests/golden/page_facts.json), torch's own float8_e4m3fn
conversion, or a brute-force nearest-value search written here.
"""
import json
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def f32(x):
    return struct.unpack("<f", struct.pack("<f", x))[0]


def test_e2m1_value_set_has_fifteen_values():
    vals = {oracle.e2m1_value(c) for c in range(16)}
    assert len(vals) == GOLDEN["e2m1_representable_values"]["count"]
    mags = sorted({abs(v) for v in vals})
    assert mags == GOLDEN["e2m1_magnitudes"]["values"]
    # code layout: bit 3 is the sign
    for c in range(8):
        assert oracle.e2m1_value(c | 8) == -oracle.e2m1_value(c) or c == 0


def test_e4m3_decode_matches_torch_float8():
    bits = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = bits.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert np.array_equal(ref[~nan], mine[~nan])
    assert max(mine[~nan]) == GOLDEN["e4m3_max"]["value"]


def _bf16_patterns():
    u = np.arange(1 << 16, dtype=np.uint32) << 16
    return u.view(np.float32)


def test_e4m3_encode_matches_torch_below_saturation():
    # contiguous blocks of float32 bit patterns in every binade from 2^-12 up to
    # the saturation region, both signs, through the oracle's bulk encoder
    blocks = []
    for e in range(127 - 12, 127 + 9):
        base = e << 23
        blocks.append((base, 1 << 17))
        blocks.append((base + (1 << 22), 1 << 15))
    blocks.append((0, 1 << 16))  # zero and the smallest subnormals
    for first, count in blocks:
        for sign in (0, 0x80000000):
            _, e4 = oracle.encode_range(sign | first, count)
            xs = (np.arange(count, dtype=np.uint64) + (sign | first)).astype(np.uint32).view(np.float32)
            keep = np.abs(xs) < 464.0
            ref = torch.from_numpy(xs[keep].copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(e4[keep], ref), hex(first)
    # scattered values through the scalar entry point
    rng = np.random.default_rng(1)
    xs = rng.standard_normal(3000).astype(np.float32) * np.float32(30.0)
    xs = xs[np.abs(xs) < 464.0]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(np.array([oracle.e4m3_encode(float(x)) for x in xs], np.uint8), ref)


def test_e4m3_encode_saturates_at_448():
    # the satfinite reading: everything at or above 448 maps to 448 (0x7E), sign kept
    for x in [448.0, 460.0, 464.0, 470.0, 1e6, float("inf")]:
        assert oracle.e4m3_encode(x) == 0x7E
        assert oracle.e4m3_encode(-x) == 0xFE


def _nearest_e2m1_bruteforce(y):
    """Nearest E2M1 code to float y: scan all codes, ties to the even code, clamp at 6."""
    sign = 8 if math.copysign(1.0, y) < 0 else 0
    a = min(abs(y), 6.0)
    best, bd = None, None
    for c in range(8):
        d = abs(oracle.e2m1_value(c) - a)
        if bd is None or d < bd or (d == bd and c % 2 == 0 and best % 2 == 1):
            best, bd = c, d
    return sign | best


def test_e2m1_encode_bruteforce():
    mags = GOLDEN["e2m1_magnitudes"]["values"]
    pts = set()
    for a, b in zip(mags, mags[1:]):
        mid = (a + b) / 2
        for x in (a, b, mid, np.nextafter(np.float32(mid), np.float32(0)),
                  np.nextafter(np.float32(mid), np.float32(10))):
            pts.add(float(np.float32(x)))
    rng = np.random.default_rng(2)
    pts |= set(float(x) for x in rng.uniform(-8, 8, 5000).astype(np.float32))
    pts |= {0.0, -0.0, 1e-30, -1e-30, 6.0, 6.5, 7.0, 100.0, -7.0}
    for x in pts:
        for s in (1.0, -1.0):
            y = float(np.float32(s * x))
            assert oracle.e2m1_encode(y) == _nearest_e2m1_bruteforce(y), y


def test_e2m1_ties_and_negative_zero():
    assert oracle.e2m1_encode(0.25) == 0        # tie 0 / 0.5 -> even (0)
    assert oracle.e2m1_encode(0.75) == 2        # tie 0.5 / 1 -> 1.0 (code 2)
    assert oracle.e2m1_encode(2.5) == 4         # tie 2 / 3 -> 2 (code 4)
    assert oracle.e2m1_encode(5.0) == 6         # tie 4 / 6 -> 4 (code 6)
    assert oracle.e2m1_encode(-0.1) == 8        # negative rounding to zero keeps its sign


def _nearest_e4m3_bruteforce(q):
    best, bd = None, None
    for b in range(0x7F):
        d = abs(oracle.e4m3_value(b) - q)
        if bd is None or d < bd or (d == bd and b % 2 == 0):
            best, bd = b, d
    return best


def test_group_quantizer_bruteforce_and_invariants():
    rng = np.random.default_rng(3)
    e2 = np.array([oracle.e2m1_value(c) for c in range(16)])
    groups = [rng.standard_normal(16).astype(np.float32) * np.float32(s)
              for s in (1e-4, 0.01, 1.0, 7.0, 300.0, 2000.0) for _ in range(40)]
    groups.append(np.zeros(16, np.float32))
    groups.append(np.full(16, 1e-6, np.float32))
    groups.append(np.array([6.0] + [0.0] * 15, np.float32))
    groups.append(np.array([2688.0] * 16, np.float32))
    for x in groups:
        codes, sb = oracle.quant_group16(x)
        amax = float(np.max(np.abs(x)))
        q = float(np.float32(np.float32(amax) / np.float32(6.0)))
        if q >= 448.0:
            assert sb == 0x7E
        else:
            assert sb == _nearest_e4m3_bruteforce(q)
        s = oracle.e4m3_value(sb)
        if s == 0.0:
            assert not codes.any()
            continue
        r = np.float32(1.0) / np.float32(s)
        for xi, c in zip(x, codes):
            y = float(np.float32(xi * r))
            assert c == _nearest_e2m1_bruteforce(y)
        dec = e2[codes] * s
        assert np.max(np.abs(dec)) <= 6.0 * s          # the group's max maps to <= 6 * scale
        # rounding error at most half the widest E2M1 gap (2) times the scale,
        # or the clipping of values the rounded-down scale pushes past 6
        assert np.max(np.abs(dec - x)) <= max(1.0 * s, amax - 6.0 * s) * (1 + 1e-6)


def test_p_level1_maximum_is_exact():
    # the row maximum of P after level 1 is 448*6 = 2688: its group's scale is 448 and its code 6
    codes, sb = oracle.quant_group16(np.array([GOLDEN["p_level1_range_max"]["value"]] + [1.0] * 15, np.float32))
    assert oracle.e4m3_value(sb) == 448.0
    assert codes[0] == 7 and oracle.e2m1_value(7) == 6.0


def test_quantize_rows_layout_against_group_loop():
    rng = np.random.default_rng(4)
    BH, N, D = 2, 37, 64
    x = torch.from_numpy(rng.standard_normal((BH, N, D)).astype(np.float32) * 3).to(torch.bfloat16)
    codes, scales = oracle.quantize_rows(x, BH, N, D)
    Np = oracle.round_up(N, 128)
    assert codes.shape == (BH, Np, D // 2) and scales.shape == (BH, Np, D // 16)
    xf = x.float().numpy()
    for bh in range(BH):
        for n in range(N):
            for g in range(D // 16):
                c, sb = oracle.quant_group16(xf[bh, n, 16 * g:16 * g + 16])
                assert scales[bh, n, g] == sb
                packed = (c[0::2] | (c[1::2] << 4)).astype(np.uint8)
                assert np.array_equal(codes[bh, n, 8 * g:8 * g + 8], packed)
    assert not codes[:, N:].any() and not scales[:, N:].any()


def test_quantize_v_is_rows_of_v_transposed():
    rng = np.random.default_rng(5)
    BH, N, D = 3, 200, 64
    v = torch.from_numpy(rng.standard_normal((BH, N, D)).astype(np.float32)).to(torch.bfloat16)
    vc, vs = oracle.quantize_v(v, BH, N, D)
    Np = oracle.round_up(N, 128)
    vt = torch.zeros((BH, D, Np), dtype=torch.bfloat16)
    vt[:, :, :N] = v.transpose(1, 2)
    # rows of V^T, quantized as Q/K rows with D' = N_pad
    rc, rs = oracle.quantize_rows(vt.reshape(1, BH * D, Np).contiguous(), 1, BH * D, Np)
    assert np.array_equal(vc.reshape(BH * D, Np // 2), rc[0, :BH * D])
    assert np.array_equal(vs.reshape(BH * D, Np // 16), rs[0, :BH * D])
