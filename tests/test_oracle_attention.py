"""Pins for the oracle's tiled FP4 attention.

The pages print no worked example, so the oracle is pinned by mathematics:

* exactly representable inputs built so that every quantization step is exact,
  where the tiled two-level algorithm must reproduce plain float64 softmax
  attention (numpy) to rounding level -- across several KV tiles with
  different row maxima, ragged N and the causal mask;
* closed forms (all keys equal, causal row 0);
* the online-softmax identity l = sum_j exp((S_j - m)/sqrt(D)) with S from a
  numpy matmul of the decoded operands;
* TILE and RUNNING level-1 modes coincide when there is one KV tile;
* both modes reproduce float64 softmax exactly on constructed inputs whose
  tiles have different maxima and whose running-maximum ratios are powers
  of two (softmax scale ln(2)/3), so RUNNING's level 1 (P2 below 2688,
  sP1 = 1/2688) is exercised where it differs from TILE's;
* the softmax scale enters only as a factor on S: attending to 2Q (whose
  quantization is Q's with every scale doubled, exactly) at scale c gives the
  same bits as attending to Q at scale 2c, and the exact path matches numpy
  softmax at any scale;
* the measured error against unquantized float64 attention on tiny shapes;
* mutation checks: plausible mistakes planted in a copy of the oracle source
  each make at least one of these pins fail.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "sage_oracle.c")


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def softmax_attention(q, k, v, causal, scale=None):
    """float64 reference: softmax(scale q k^T) v for [BH,N,D] arrays (scale 1/sqrt(D))."""
    BH, N, D = q.shape
    s = np.einsum("bid,bjd->bij", q, k) * (1.0 / np.sqrt(D) if scale is None else scale)
    if causal:
        s = np.where(np.tril(np.ones((N, N), bool))[None], s, -np.inf)
    s = s - s.max(-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(-1, keepdims=True)
    return np.einsum("bij,bjd->bid", p, v)


def exact_case(BH, N, D, seed, hit_choices=(6.0, 4.0, 3.0, 2.0, 1.5)):
    """Inputs on which the oracle's quantization is exact.

    Each 16-element group holds values of the E2M1 grid with one element of
    magnitude 6, so its scale is a power of two.  Scores: q = [6 or 3, 0, 6, ..| 96, ..],
    and each key is a "hit" (S = 6*k0 or 3*k0, the same for every hit of a KV
    tile) or a "miss" (S far below the hits).  The
    first key of every tile is a hit, so every row's tile maximum is a hit and
    level-1/level-2 quantization of P is exact ({2688, ~0}).
    """
    assert D >= 64
    rng = np.random.default_rng(seed)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    q = np.zeros((BH, N, D))
    q[:, :, 0] = rng.choice([6.0, 3.0], size=(BH, N))
    q[:, :, 2] = 6.0
    q[:, :, 16] = 96.0  # group 1 = [96, 0, ...]: scale 16 (exact), code 6
    k = np.zeros((BH, N, D))
    k[:, :, 1] = 6.0
    ntile = (N + 127) // 128
    hit_vals = rng.choice(list(hit_choices), size=(BH, ntile))
    hit = rng.random((BH, N)) < 0.35
    hit[:, ::128] = True
    for t in range(ntile):
        sl = slice(128 * t, min(N, 128 * t + 128))
        k[:, sl, 0] = np.where(hit[:, sl], hit_vals[:, t:t + 1], rng.choice(grid, size=hit[:, sl].shape))
        k[:, sl, 16] = np.where(hit[:, sl], 0.0, -6.0)
    v = rng.choice(grid, size=(BH, N, D)) * rng.choice([-1.0, 1.0], size=(BH, N, D))
    v[:, ::16, :] = 6.0 * rng.choice([-1.0, 1.0], size=v[:, ::16, :].shape)
    return q, k, v


def run_oracle(q, k, v, causal, pmode="tile", rows=None):
    BH, N, D = q.shape
    qz = oracle.Quantized(bf16(q), bf16(k), bf16(v), BH, N, D)
    return oracle.attention(qz, causal, pmode, rows=rows), qz


@pytest.mark.parametrize("N,causal", [(300, False), (300, True), (128, False), (513, True)])
def test_exactly_quantizable_inputs_reproduce_softmax(N, causal):
    BH, D = 2, 64
    q, k, v = exact_case(BH, N, D, seed=N + causal)
    (o, l, m), qz = run_oracle(q, k, v, causal)
    # quantization is the identity on these inputs
    assert np.array_equal(oracle.decode_rows(qz.qc, qz.qs)[:, :N], q)
    assert np.array_equal(oracle.decode_rows(qz.kc, qz.ks)[:, :N], k)
    assert np.array_equal(oracle.decode_rows(qz.vc, qz.vs)[:, :, :N], v.transpose(0, 2, 1))
    ref = softmax_attention(q, k, v, causal).reshape(BH * N, D)
    err = np.abs(o - ref).max() / np.abs(ref).max()
    assert err < 1e-12, err


# Level 1 in RUNNING mode maps each tile against the running maximum m, so a
# tile whose maximum t lies below m gets P2 = 2688 * exp((t - m) * scale) < 2688
# and sP1 = 1/2688.  With hit scores q0 * h, q0 in {3, 6} and h in {6, 4, 3, 2},
# every difference t - m within a row is a multiple of 3; at the softmax scale
# ln(2)/3 each exp((t - m) * scale) is a power of two 2^-k (k <= 8), so P2 of a
# hit is 2688 * 2^-k: an exact E4M3 scale 448 * 2^-k with code 6.  Quantization
# of P stays exact in both modes, tiles have different maxima, and both modes
# must reproduce float64 softmax attention at that scale.
RUNNING_SCALE = np.log(2.0) / 3.0


@pytest.mark.parametrize("pmode", ["tile", "running"])
@pytest.mark.parametrize("N,causal", [(513, False), (513, True), (300, False)])
def test_exactly_quantizable_inputs_with_differing_tile_maxima(N, causal, pmode):
    BH, D = 2, 64
    q, k, v = exact_case(BH, N, D, seed=3 * N + causal, hit_choices=(6.0, 4.0, 3.0, 2.0))
    qz = oracle.Quantized(bf16(q), bf16(k), bf16(v), BH, N, D)
    o, l, m = oracle.attention(qz, causal, pmode, scale=RUNNING_SCALE)
    ref = softmax_attention(q, k, v, causal, scale=RUNNING_SCALE).reshape(BH * N, D)
    err = np.abs(o - ref).max() / np.abs(ref).max()
    assert err < 1e-12, (pmode, err)
    if not causal:
        # the case does what it is for: some rows see a later tile whose
        # maximum exceeds every earlier one, and later tiles whose maximum is
        # below the running one (where RUNNING's level 1 differs from TILE's)
        qd = oracle.decode_rows(qz.qc, qz.qs)[:, :N]
        kd = oracle.decode_rows(qz.kc, qz.ks)[:, :N]
        s = np.einsum("bid,bjd->bij", qd, kd)
        ntile = (N + 127) // 128
        tmax = np.stack([s[:, :, 128 * t:128 * t + 128].max(-1) for t in range(ntile)], -1)
        running = np.maximum.accumulate(tmax, axis=-1)
        assert (tmax[..., 1:] < running[..., 1:]).any()
        assert (tmax[..., 1:] > running[..., :-1]).any()


def decoded(qz):
    N = qz.N
    qd = oracle.decode_rows(qz.qc, qz.qs)[:, :N]
    kd = oracle.decode_rows(qz.kc, qz.ks)[:, :N]
    vd = oracle.decode_rows(qz.vc, qz.vs)[:, :, :N].transpose(0, 2, 1)
    return qd, kd, vd


@pytest.mark.parametrize("causal", [False, True])
def test_all_keys_equal_gives_mean_of_decoded_v(causal):
    BH, N, D = 2, 300, 128
    rng = np.random.default_rng(7)
    q = rng.standard_normal((BH, N, D)) * 2
    k = np.repeat(rng.standard_normal((BH, 1, D)), N, axis=1)
    v = rng.standard_normal((BH, N, D))
    (o, l, m), qz = run_oracle(q, k, v, causal)
    _, _, vd = decoded(qz)
    if causal:
        ref = np.cumsum(vd, axis=1) / np.arange(1, N + 1)[None, :, None]
    else:
        ref = np.repeat(vd.mean(axis=1, keepdims=True), N, axis=1)
    assert np.abs(o - ref.reshape(BH * N, D)).max() < 1e-12


def test_zero_q_gives_mean_of_decoded_v():
    BH, N, D = 1, 200, 64
    rng = np.random.default_rng(8)
    (o, _, _), qz = run_oracle(np.zeros((BH, N, D)), rng.standard_normal((BH, N, D)) * 5,
                               rng.standard_normal((BH, N, D)), False)
    _, _, vd = decoded(qz)
    assert np.abs(o - vd.mean(axis=1)).max() < 1e-12


def test_causal_row_zero_is_first_value_row():
    BH, N, D = 3, 150, 128
    rng = np.random.default_rng(9)
    rows = [bh * N for bh in range(BH)]
    (o, _, _), qz = run_oracle(rng.standard_normal((BH, N, D)) * 3, rng.standard_normal((BH, N, D)),
                               rng.standard_normal((BH, N, D)), True, rows=rows)
    _, _, vd = decoded(qz)
    assert np.array_equal(o, vd[:, 0, :])


@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_row_statistics(causal):
    """m is the row max of S = Q^ K^T (numpy matmul of the decoded operands), and
    l equals sum_j exp((S_j - m)/sqrt(D)): the unquantized probabilities divided by
    l sum to one."""
    from bit_attention_gb300.synth import make_qkv
    B, H, N, D = 1, 2, 333, 128
    q, k, v = make_qkv(B, H, N, D, "k_channel_outliers", seed=3)
    qz = oracle.Quantized(q, k, v, B * H, N, D)
    o, l, m = oracle.attention(qz, causal)
    qd, kd, _ = decoded(qz)
    s = np.einsum("bid,bjd->bij", qd, kd)
    if causal:
        s = np.where(np.tril(np.ones((N, N), bool))[None], s, -np.inf)
    m_ref = s.max(-1).reshape(-1)
    assert np.allclose(m, m_ref, rtol=1e-13, atol=1e-9)
    p = np.exp((s - m_ref.reshape(B * H, N, 1)) / np.sqrt(D))
    rowsum = p.sum(-1).reshape(-1) / l
    assert np.abs(rowsum - 1.0).max() < 1e-12


def test_tile_and_running_modes_agree_on_one_tile():
    rng = np.random.default_rng(10)
    BH, N, D = 2, 100, 64
    q, k, v = (rng.standard_normal((BH, N, D)) * s for s in (1, 3, 1))
    qz = oracle.Quantized(bf16(q), bf16(k), bf16(v), BH, N, D)
    for causal in (False, True):
        a = oracle.attention(qz, causal, "tile")[0]
        b = oracle.attention(qz, causal, "running")[0]
        assert np.array_equal(a, b)


# measured (cosine, relative L1) of the oracle against exact attention, seed 11,
# both level-1 modes: iid 0.984/0.179, iid causal D64 0.986/0.174,
# K channel outliers 0.842/0.542, K head mean D64 0.966/0.260.  The bounds
# below add headroom; K outlier channels cost the most (no K smoothing).
UNQUANTIZED_CASES = {
    "iid": (("iid", 256, 128, False), 0.975, 0.22),
    "iid_causal_d64": (("iid", 200, 64, True), 0.975, 0.22),
    "k_outliers": (("k_channel_outliers", 384, 128, False), 0.82, 0.58),
    "k_head_mean_d64": (("k_head_mean", 300, 64, False), 0.955, 0.30),
}


@pytest.mark.parametrize("case", sorted(UNQUANTIZED_CASES))
def test_against_unquantized_attention(case):
    """Self-check against exact float64 attention on tiny shapes (the pages give
    no error bound; these are measured bounds with headroom)."""
    from bit_attention_gb300.synth import make_qkv
    (pattern, N, D, causal), cos_min, rel_max = UNQUANTIZED_CASES[case]
    q, k, v = make_qkv(1, 2, N, D, pattern, seed=11)
    qz = oracle.Quantized(q, k, v, 2, N, D)
    ref = oracle.attention_exact(q, k, v, 2, N, D, causal)
    ref_np = softmax_attention(*(t.float().numpy().reshape(2, N, D).astype(np.float64)
                                 for t in (q, k, v)), causal)
    assert np.abs(ref - ref_np.reshape(-1, D)).max() < 1e-10
    for pmode in ("tile", "running"):
        o = oracle.attention(qz, causal, pmode)[0]
        cos = (o * ref).sum() / np.sqrt((o * o).sum() * (ref * ref).sum())
        rel_l1 = np.abs(o - ref).sum() / np.abs(ref).sum()
        assert cos >= cos_min and rel_l1 <= rel_max, (pmode, cos, rel_l1)


@pytest.mark.parametrize("D,causal", [(64, False), (128, True)])
def test_scale_is_a_factor_on_scores(D, causal):
    """Q -> 2Q doubles every E4M3 scale of Q exactly and keeps its codes, so S
    doubles exactly; attention at scale c on 2Q must equal attention at scale
    2c on Q bit for bit, in the tiled and in the exact oracle."""
    from bit_attention_gb300.synth import make_qkv
    BH, N = 2, 300
    q, k, v = make_qkv(1, BH, N, D, "iid", seed=5)
    q2 = (q.float() * 2).to(torch.bfloat16)
    qz, qz2 = oracle.Quantized(q, k, v, BH, N, D), oracle.Quantized(q2, k, v, BH, N, D)
    assert np.array_equal(qz.qc, qz2.qc)
    e4 = np.array([oracle.e4m3_value(b) for b in range(256)])
    assert np.array_equal(e4[qz2.qs], 2 * e4[qz.qs])
    c = 1.0 / np.sqrt(D)
    o_twice_q = oracle.attention(qz2, causal, scale=c)[0]
    o_twice_scale = oracle.attention(qz, causal, scale=2 * c)[0]
    assert np.array_equal(o_twice_q, o_twice_scale)
    assert not np.array_equal(o_twice_scale, oracle.attention(qz, causal)[0])
    e_twice_q = oracle.attention_exact(q2, k, v, BH, N, D, causal, scale=c)
    e_twice_scale = oracle.attention_exact(q, k, v, BH, N, D, causal, scale=2 * c)
    assert np.array_equal(e_twice_q, e_twice_scale)


@pytest.mark.parametrize("scale", [0.03, 0.5])
def test_exact_attention_matches_numpy_at_any_scale(scale):
    from bit_attention_gb300.synth import make_qkv
    BH, N, D = 2, 200, 64
    q, k, v = make_qkv(1, BH, N, D, "iid", seed=9)
    got = oracle.attention_exact(q, k, v, BH, N, D, True, scale=scale)
    want = softmax_attention(*(t.float().numpy().reshape(BH, N, D).astype(np.float64) for t in (q, k, v)),
                             True, scale=scale)
    assert np.abs(got - want.reshape(-1, D)).max() < 1e-10


# ---------------------------------------------------------------- mutations
MUTATIONS = {
    "drop_alpha": ("acc[d] = acc[d] * alpha + sP1 * pv;", "acc[d] = acc[d] + sP1 * pv;"),
    "drop_sP1": ("acc[d] = acc[d] * alpha + sP1 * pv;", "acc[d] = acc[d] * alpha + pv / 2688.0;"),
    "l_not_rescaled": ("l = l * alpha + lt;", "l = l + lt;"),
    "exp_sign": ("P2[jj] = (float)(R * exp((S[jj] - ref) * isd));",
                 "P2[jj] = (float)(R * exp((ref - S[jj]) * isd));"),
    "k_scale_index": ("sc[ks[(size_t)j * G + g]]", "sc[ks[(size_t)i * G + g]]"),
    "v_group_index": ("sc[vsrow[jg]]", "sc[vsrow[g]]"),
    "causal_off_by_one": ("int kend = causal ? (i + 1) : N;", "int kend = causal ? i : N;"),
    "no_level2_scale": ("pv += sc[ps[g]] * sc[vsrow[jg]] * part;",
                        "pv += 448.0 * sc[vsrow[jg]] * part;"),
    "scale_amax_over_4": ("float q = amax / 6.0f;", "float q = amax / 4.0f;"),
    "e2m1_ties_up": ("(d == bestd && (i & 1) == 0)", "(d == bestd)"),
    "l_against_tile_max": ("lt += exp((S[jj] - m_new) * isd);", "lt += exp((S[jj] - t) * isd);"),
    "nibble_order": ("  if (idx & 1)\n    row[idx >> 1] = (uint8_t)((row[idx >> 1] & 0x0F) | (code << 4));",
                     "  if (!(idx & 1))\n    row[idx >> 1] = (uint8_t)((row[idx >> 1] & 0x0F) | (code << 4));"),
    "dot_drops_element": ("for (int k = GS * g; k < GS * g + GS; k++)", "for (int k = GS * g + 1; k < GS * g + GS; k++)"),
    "e4m3_subnormal_step": ("return sign | (int)rint(a * 512.0);", "return sign | (int)rint(a * 256.0);"),
    "running_sP1_as_tile": ("double sP1 = (pmode == 0) ? exp((t - m_new) * isd) / R : 1.0 / R;",
                            "double sP1 = exp((t - m_new) * isd) / R;"),
    "running_ref_is_tile_max": ("double ref = (pmode == 0) ? t : m_new;", "double ref = t;"),
    "directp_drops_group_scale": ("        rounded += sc[ps[g]] * part;", "        rounded += part;"),
    "directp_omits_sP1": ("      lt = sP1 * rounded;", "      lt = rounded / R;"),
    "directp_normaliser_unused": ("    if (lnorm == 1) {", "    if (lnorm == 2) {"),
    "directp_drops_code": ("for (int k = 0; k < GS; k++) part += g_e2m1[pc[GS * g + k]];",
                           "for (int k = 1; k < GS; k++) part += g_e2m1[pc[GS * g + k]];"),
    "scale_ignored": ("double *out_m) {\n  const double isd = scale;",
                      "double *out_m) {\n  const double isd = 1.0 / sqrt((double)D);"),
}


def all_pins():
    """Run the pins above; return the names of the ones that fail."""
    failed = []
    checks = [
        ("exact_noncausal", lambda: test_exactly_quantizable_inputs_reproduce_softmax(300, False)),
        ("exact_causal", lambda: test_exactly_quantizable_inputs_reproduce_softmax(300, True)),
        ("equal_k", lambda: test_all_keys_equal_gives_mean_of_decoded_v(True)),
        ("row0", test_causal_row_zero_is_first_value_row),
        ("rowstats", lambda: test_online_softmax_row_statistics(False)),
        ("codec_ties", lambda: __import__("test_oracle_codecs").test_e2m1_ties_and_negative_zero()),
        ("group", lambda: __import__("test_oracle_codecs").test_group_quantizer_bruteforce_and_invariants()),
        ("unquantized", lambda: test_against_unquantized_attention("iid")),
        ("scale", lambda: test_scale_is_a_factor_on_scores(64, False)),
        ("exact_running", lambda: test_exactly_quantizable_inputs_with_differing_tile_maxima(
            513, False, "running")),
        ("directp_exact", lambda: __import__("test_oracle_directp")
         .test_exactly_quantizable_mx_inputs_give_softmax_with_either_normaliser(513, False)),
        ("directp_two_keys", lambda: __import__("test_oracle_directp").test_two_visible_keys_closed_form("mxfp4")),
        ("directp_constant_v", lambda: __import__("test_oracle_directp")
         .test_constant_v_is_returned_exactly("mxfp4", False)),
    ]
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
        except Exception:
            failed.append(name)
    return failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, name
    mutated = tmp_path / "sage_oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "sage_oracle.h").write_text(open(ORACLE_SRC[:-2] + ".h").read())
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    str(mutated), "-o", str(so), "-lm"], check=True)
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    with oracle.swapped(str(so)):
        failed = all_pins()
    assert failed, f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_all_pins():
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    assert all_pins() == []
