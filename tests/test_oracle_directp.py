"""Pins for the oracle's Direct-P normaliser (lnorm="rounded").

Direct-P (the rit.work summary of "Hardware-Aware FP4 FlashAttention-4",
"Что сделали") sums the softmax normaliser from the same rounded
probabilities that enter PV, instead of from the unquantized exponentials.
The pins:

* exactly quantizable MXFP4 inputs (tiles with different maxima, 32-key
  groups whose scale is 1/2): P quantization is exact, so both normalisers
  give float64 softmax attention;
* a causal row with two visible keys whose P2 values are 6 and 2.7: 2.7
  rounds to 3, so Direct-P gives O = (6 v0 + 3 v1) / 9 exactly (the
  unquantized normaliser gives (6 v0 + 3 v1) / 8.7);
* V constant along tokens: PV and l use the same rounded P, so Direct-P
  returns that constant exactly, where the unquantized normaliser does not.
"""
import numpy as np
import pytest
import torch

import oracle

LN2_OVER_3 = np.log(2.0) / 3.0


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def softmax_attention(q, k, v, causal, scale):
    BH, N, D = q.shape
    s = np.einsum("bid,bjd->bij", q, k) * scale
    if causal:
        s = np.where(np.tril(np.ones((N, N), bool))[None], s, -np.inf)
    s = s - s.max(-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(-1, keepdims=True)
    return np.einsum("bij,bjd->bid", p, v)


def exact_mx_case(BH, N, seed):
    """MXFP4-exact inputs, D = 64 (two 32-element groups along D).

    q = [3, 0, 6, 0...| 96, 0...]: group scales 1 and 16, codes exact.
    k = [h, 6, 0...| 0 or -6, 0...]: S = 3 h for a hit, 3 h - 576 for a miss.
    In every KV tile the first key is a full hit (h = hv), keys 32-63 hold
    only half hits (h = hv - 1, S three lower) and misses, the rest a mix.
    At softmax scale ln(2)/3 a full hit has P2 = 6 (scale 1, code 6), a half
    hit P2 = 3 (scale 1, or 1/2 with code 6 in a group without full hits), a
    miss P2 = 0: every quantization step is exact."""
    D = 64
    rng = np.random.default_rng(seed)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    q = np.zeros((BH, N, D))
    q[:, :, 0] = 3.0
    q[:, :, 2] = 6.0
    q[:, :, 32] = 96.0
    k = np.zeros((BH, N, D))
    k[:, :, 1] = 6.0
    ntile = (N + 127) // 128
    hv = rng.choice([4.0, 3.0, 2.0], size=(BH, ntile))
    for b in range(BH):
        for t in range(ntile):
            for jj in range(min(128, N - 128 * t)):
                j = 128 * t + jj
                u = rng.random()
                if jj == 0 or (jj >= 64 and u < 0.25) or (jj < 32 and u < 0.3):
                    k[b, j, 0] = hv[b, t]                       # full hit
                elif 32 <= jj < 64 and u < 0.35 or jj >= 64 and u < 0.5:
                    k[b, j, 0] = hv[b, t] - 1.0                 # half hit
                else:
                    k[b, j, 0] = rng.choice(grid)               # miss
                    k[b, j, 32] = -6.0
    v = rng.choice(grid, size=(BH, N, D)) * rng.choice([-1.0, 1.0], size=(BH, N, D))
    v[:, ::32, :] = 6.0 * rng.choice([-1.0, 1.0], size=v[:, ::32, :].shape)
    return q, k, v


@pytest.mark.parametrize("N,causal", [(300, False), (513, False), (257, True)])
def test_exactly_quantizable_mx_inputs_give_softmax_with_either_normaliser(N, causal):
    BH = 2
    q, k, v = exact_mx_case(BH, N, seed=N + causal)
    qz = oracle.Quantized(bf16(q), bf16(k), bf16(v), BH, N, 64, fmt="mxfp4")
    assert np.array_equal(oracle.decode_rows(qz.qc, qz.qs, "mxfp4")[:, :N], q)
    assert np.array_equal(oracle.decode_rows(qz.kc, qz.ks, "mxfp4")[:, :N], k)
    ref = softmax_attention(q, k, v, causal, LN2_OVER_3).reshape(BH * N, 64)
    outs = {}
    for ln in ("exp", "rounded"):
        o, l, _ = oracle.attention(qz, causal, scale=LN2_OVER_3, lnorm=ln)
        assert np.abs(o - ref).max() / np.abs(ref).max() < 1e-12, ln
        outs[ln] = l
    assert np.allclose(outs["exp"], outs["rounded"], rtol=1e-13, atol=0)


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_two_visible_keys_closed_form(fmt):
    """Row 1 of a causal head sees keys 0 and 1 with S = 12 and 9.  At the
    softmax scale ln(1/0.45)/3 their level-1 values are R and 0.45 R; in the
    row's group (maximum R: scale 1 for MXFP4, 448 for NVFP4) 0.45 R decodes
    to 3/6 R, so Direct-P weighs V0 and V1 as 6 : 3."""
    BH, N, D = 1, 40, 64
    scale = np.log(1 / 0.45) / 3.0
    rng = np.random.default_rng(3)
    q = np.zeros((BH, N, D))
    q[:, :, 0] = 3.0
    q[:, :, 2] = 6.0
    k = np.zeros((BH, N, D))
    k[:, :, 1] = 6.0
    k[:, 0, 0] = 4.0
    k[:, 1, 0] = 3.0
    k[:, 2:, 0] = rng.choice([0.5, 1.0, 2.0], size=(BH, N - 2))
    v = rng.standard_normal((BH, N, D))
    qz = oracle.Quantized(bf16(q), bf16(k), bf16(v), BH, N, D, fmt=fmt)
    vd = oracle.decode_rows(qz.vc, qz.vs, fmt)[:, :, :N].transpose(0, 2, 1)
    want = (6.0 * vd[0, 0] + 3.0 * vd[0, 1]) / 9.0
    o, l, _ = oracle.attention(qz, True, rows=[1], scale=scale, lnorm="rounded")
    assert np.abs(o[0] - want).max() <= 1e-12 * np.abs(want).max()
    o_exp = oracle.attention(qz, True, rows=[1], scale=scale, lnorm="exp")[0]
    assert np.abs(o_exp[0] - (6.0 * vd[0, 0] + 3.0 * vd[0, 1]) / 8.7).max() <= 1e-6 * np.abs(want).max()


@pytest.mark.parametrize("fmt,causal", [("mxfp4", False), ("mxfp4", True), ("nvfp4", False)])
def test_constant_v_is_returned_exactly(fmt, causal):
    from bit_attention_gb300.synth import make_qkv
    BH, N, D = 2, 333, 128
    q, k, _ = make_qkv(1, BH, N, D, "k_channel_outliers", seed=8)
    v = torch.full((1, BH, N, D), 1.5, dtype=torch.bfloat16)
    qz = oracle.Quantized(q, k, v, BH, N, D, fmt=fmt)
    o = oracle.attention(qz, causal, lnorm="rounded")[0]
    assert np.abs(o - 1.5).max() < 1e-12
    o_exp = oracle.attention(qz, causal, lnorm="exp")[0]
    assert np.abs(o_exp - 1.5).max() > 1e-4   # the unquantized normaliser leaves a bias


def test_rounded_normaliser_changes_o_on_random_inputs():
    from bit_attention_gb300.synth import make_qkv
    BH, N, D = 2, 300, 128
    q, k, v = make_qkv(1, BH, N, D, "iid", seed=9)
    qz = oracle.Quantized(q, k, v, BH, N, D, fmt="mxfp4")
    a, la, _ = oracle.attention(qz, False, lnorm="exp")
    b, lb, _ = oracle.attention(qz, False, lnorm="rounded")
    assert not np.array_equal(a, b)
    assert np.abs(lb / la - 1).max() < 0.2      # the same normaliser up to P rounding
    with pytest.raises(KeyError):
        oracle.attention(qz, False, lnorm="other")
