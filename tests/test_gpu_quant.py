"""Quantize kernel parity: codes and scales bit-exact with the oracle.

Shapes span several 128-row tiles and ragged tails (N not a multiple of 16 or
128), both head dims and the workloads' value patterns; every benchmark
workload (up to B4 H32 N8192 D128 and B2 H48 N17776 D64) is compared in full,
in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300.synth import WORKLOADS, make_qkv
from helpers import block_to_plain

pytestmark = pytest.mark.gpu


def check_quant(q, k, v):
    B, H, N, D = q.shape
    BH = B * H
    z = S.quantize_qkv(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    Np = z.Np
    for name, x, codes, scales in (("q", q, z.q_codes, z.q_scales), ("k", k, z.k_codes, z.k_scales)):
        rc, rs = oracle.quantize_rows(x, BH, N, D)
        gc = codes.cpu().numpy()
        gs = block_to_plain(scales.cpu().numpy(), Np, D // 16)
        assert np.array_equal(gc, rc), f"{name} codes differ at {np.argwhere(gc != rc)[:5]}"
        assert np.array_equal(gs, rs), f"{name} scales differ at {np.argwhere(gs != rs)[:5]}"
    rc, rs = oracle.quantize_v(v, BH, N, D)
    gc = z.vt_codes.cpu().numpy()
    gs = block_to_plain(z.vt_scales.cpu().numpy(), 128, Np // 16)
    assert np.array_equal(gc, rc), f"vt codes differ at {np.argwhere(gc != rc)[:5]}"
    assert np.array_equal(gs[:, :D], rs), f"vt scales differ at {np.argwhere(gs[:, :D] != rs)[:5]}"
    assert not gs[:, D:].any()
    return z


@pytest.mark.parametrize("B,H,N,D,pattern", [
    (1, 2, 512, 128, "iid"),
    (2, 3, 200, 64, "iid"),
    (1, 1, 17, 128, "iid"),
    (1, 2, 1000, 128, "k_channel_outliers"),
    (2, 2, 130, 64, "k_head_mean"),
    (1, 3, 777, 128, "sparse_outliers"),
    (1, 1, 1, 64, "iid"),
])
def test_quantize_bit_exact(B, H, N, D, pattern):
    q, k, v = make_qkv(B, H, N, D, pattern, seed=N)
    check_quant(q, k, v)


def test_quantize_special_values():
    # zeros, tiny values whose scale rounds to zero, negative values that round
    # to zero (-0 code), exact maxima, large values up to the E4M3 saturation
    B, H, N, D = 1, 1, 256, 128
    rng = np.random.default_rng(0)
    x = rng.standard_normal((B, H, N, D)).astype(np.float32)
    x[0, 0, 0] = 0.0
    x[0, 0, 1] = 1e-5 * rng.standard_normal(D)
    x[0, 0, 2, :16] = -1e-3
    x[0, 0, 2, 0] = 6.0
    x[0, 0, 3] = 3000.0 * rng.standard_normal(D)
    x[0, 0, 4] = np.tile(np.array([6.0, 4.0, 3.0, 2.0, 1.5, 1.0, 0.5, 0.25] * 2, np.float32), D // 16)
    x[0, 0, 5] = -x[0, 0, 4] * 0.75
    t = torch.from_numpy(x).to(torch.bfloat16)
    check_quant(t, t.clone(), t.clone())


@pytest.mark.parametrize("name", ["small", "llm", "llm_causal", "dit", "dit_long"])
def test_quantize_full_workload(name):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.pattern, seed=0)
    check_quant(q, k, v)


def test_every_bf16_magnitude_as_group_absmax():
    # Every non-negative finite bf16 value (bit patterns 0x0000-0x7F7F, 32640
    # of them, subnormals included) is the absmax of exactly one group, in Q
    # and K (groups along D) and in V (groups along tokens).  The kernels take
    # amax/6 as amax*RN(1/6) plus one FMA residual step, which must equal the
    # correctly rounded quotient the oracle computes for every one of them;
    # the other 15 elements of a group are random fractions of its absmax, of
    # either sign, so the codes are checked across the whole range as well.
    amax = (np.arange(0x7F80, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    G = amax.size
    rng = np.random.default_rng(4)
    frac = rng.uniform(-1.0, 1.0, size=(G, 16))
    frac[np.arange(G), rng.integers(0, 16, size=G)] = rng.choice([-1.0, 1.0], size=G)
    # float64 -> float32 -> bf16, each rounding to nearest: |x| <= amax stays true
    groups = torch.from_numpy((amax[:, None] * frac).astype(np.float32)).to(torch.bfloat16)
    got_amax = groups.float().abs().amax(1).numpy()
    assert np.array_equal(got_amax, amax.astype(np.float32))
    D, N = 128, G * 16 // 128  # 4080 rows of 8 groups
    q = groups.reshape(1, 1, N, D)
    k = q.flip(2).contiguous()
    # V: group g of channel d is tokens 16g..16g+15 of channel d
    v = groups.reshape(D, N // 16, 16).reshape(D, N).t().contiguous().reshape(1, 1, N, D)
    check_quant(q, k, v)
