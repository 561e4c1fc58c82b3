"""Pins for the oracle's MXFP4 variant (1x32 groups, E8M0 scales).

The pages weigh MXFP4 against NVFP4 and keep NVFP4 for its accuracy
([NEWS-HW]); the MXFP4 variant of the method swaps the microscaling format in
every quantization step.  The pages fix the format, not the rounding rule;
the oracle follows the OCP MX v1.0 conversion (shared exponent floor(log2
amax) - 2, elements x / 2^shared rounded to nearest E2M1).  Pinned by:

* E8M0 structure: byte 127 is 1, each byte doubles the one below, 0xFF is NaN;
* the group quantizer against a brute force: the scale is the power of two X
  with 4 <= amax / X < 8, and each code is the E2M1 value nearest x / X (ties
  to even, saturating at 6);
* exactly representable inputs (every 32-element group's maximum is 6 x 2^k,
  the rest on the E2M1 grid at that power), where the tiled MXFP4 attention
  must reproduce float64 softmax attention to rounding;
* the closed forms (all keys equal: mean of the decoded V; causal row 0);
* planted mistakes (scale exponent off by one, NVFP4's level-1 target) fail
  one of these.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle

sys.path.insert(0, os.path.dirname(__file__))
from test_oracle_attention import ORACLE_SRC, bf16, softmax_attention  # noqa: E402
from test_oracle_codecs import _nearest_e2m1_bruteforce  # noqa: E402


def test_e8m0_structure():
    assert oracle.e8m0_value(127) == 1.0
    for b in range(254):
        assert oracle.e8m0_value(b + 1) == 2 * oracle.e8m0_value(b)
    assert oracle.e8m0_value(0) > 0 and np.isnan(oracle.e8m0_value(255))


def test_mx_group_quantizer_bruteforce():
    rng = np.random.default_rng(13)
    groups = [rng.standard_normal(32).astype(np.float32) * np.float32(s)
              for s in (1e-30, 1e-4, 0.3, 1.0, 7.0, 300.0, 1e20) for _ in range(30)]
    groups += [np.zeros(32, np.float32), np.array([6.0] + [0.0] * 31, np.float32),
               np.array([4.0] + [-7.99] * 31, np.float32), np.array([8.0, 5.0, 3.5, 0.25] * 8, np.float32)]
    for x in groups:
        codes, sb = oracle.quant_group32_mx(x)
        amax = float(np.max(np.abs(x)))
        X = oracle.e8m0_value(sb)
        if amax == 0.0:
            assert sb == 0 and all(c & 7 == 0 for c in codes)
            continue
        assert 4.0 <= amax / X < 8.0, (amax, X)
        for xi, c in zip(x, codes):
            assert c == _nearest_e2m1_bruteforce(float(xi) / X), (xi, X, c)


def test_mx_level1_maximum_is_exact():
    # after level 1 the tile's row maximum is 6: scale 2^0 (byte 127), code 6
    codes, sb = oracle.quant_group32_mx(np.array([6.0] + [0.5] * 31, np.float32))
    assert sb == 127 and codes[0] == 7


def exact_case_mx(BH, N, D, seed):
    """Inputs on which MXFP4 quantization is the identity (groups of 32).

    Scores as in the NVFP4 exact case (each key a "hit", with the tile's
    common score, or a "miss" far below), with the large element of q and the
    miss marker of k moved to channel 32, the start of the second group."""
    assert D >= 64
    rng = np.random.default_rng(seed)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    q = np.zeros((BH, N, D))
    q[:, :, 0] = rng.choice([6.0, 3.0], size=(BH, N))
    q[:, :, 2] = 6.0
    q[:, :, 32] = 96.0  # group 1 = [96, 0, ...]: scale 16, code 6
    k = np.zeros((BH, N, D))
    k[:, :, 1] = 6.0
    ntile = (N + 127) // 128
    hit_vals = rng.choice([6.0, 4.0, 3.0, 2.0, 1.5], size=(BH, ntile))
    hit = rng.random((BH, N)) < 0.35
    hit[:, ::128] = True
    for t in range(ntile):
        sl = slice(128 * t, min(N, 128 * t + 128))
        k[:, sl, 0] = np.where(hit[:, sl], hit_vals[:, t:t + 1], rng.choice(grid, size=hit[:, sl].shape))
        k[:, sl, 32] = np.where(hit[:, sl], 0.0, -6.0)
    v = rng.choice(grid, size=(BH, N, D)) * rng.choice([-1.0, 1.0], size=(BH, N, D))
    v[:, ::32, :] = 6.0 * rng.choice([-1.0, 1.0], size=v[:, ::32, :].shape)
    return q, k, v


def run_mx(q, k, v, causal, rows=None):
    BH, N, D = q.shape
    qz = oracle.Quantized(bf16(q), bf16(k), bf16(v), BH, N, D, fmt="mxfp4")
    return oracle.attention(qz, causal, rows=rows), qz


def decoded_mx(qz):
    N = qz.N
    return (oracle.decode_rows(qz.qc, qz.qs, "mxfp4")[:, :N], oracle.decode_rows(qz.kc, qz.ks, "mxfp4")[:, :N],
            oracle.decode_rows(qz.vc, qz.vs, "mxfp4")[:, :, :N].transpose(0, 2, 1))


@pytest.mark.parametrize("N,causal", [(300, False), (300, True), (513, True)])
def test_mx_exactly_quantizable_inputs_reproduce_softmax(N, causal):
    BH, D = 2, 64
    q, k, v = exact_case_mx(BH, N, D, seed=N + causal)
    (o, _, _), qz = run_mx(q, k, v, causal)
    qd, kd, vd = decoded_mx(qz)
    assert np.array_equal(qd, q) and np.array_equal(kd, k) and np.array_equal(vd, v)
    ref = softmax_attention(q, k, v, causal).reshape(BH * N, D)
    err = np.abs(o - ref).max() / np.abs(ref).max()
    assert err < 1e-12, err


@pytest.mark.parametrize("causal", [False, True])
def test_mx_all_keys_equal_gives_mean_of_decoded_v(causal):
    BH, N, D = 2, 300, 128
    rng = np.random.default_rng(7)
    q = rng.standard_normal((BH, N, D)) * 2
    k = np.repeat(rng.standard_normal((BH, 1, D)), N, axis=1)
    v = rng.standard_normal((BH, N, D))
    (o, _, _), qz = run_mx(q, k, v, causal)
    vd = decoded_mx(qz)[2]
    if causal:
        ref = np.cumsum(vd, axis=1) / np.arange(1, N + 1)[None, :, None]
    else:
        ref = np.repeat(vd.mean(axis=1, keepdims=True), N, axis=1)
    assert np.abs(o - ref.reshape(BH * N, D)).max() < 1e-12


def test_mx_causal_row_zero_is_first_value_row():
    BH, N, D = 3, 150, 128
    rng = np.random.default_rng(9)
    rows = [bh * N for bh in range(BH)]
    (o, _, _), qz = run_mx(rng.standard_normal((BH, N, D)) * 3, rng.standard_normal((BH, N, D)),
                           rng.standard_normal((BH, N, D)), True, rows=rows)
    assert np.array_equal(o, decoded_mx(qz)[2][:, 0, :])


MX_MUTATIONS = {
    "mx_emax_1": ("int shared = (E - 1) - 2;", "int shared = (E - 1) - 1;"),
    "mx_level1_2688": ("const double R = (fmt == SOR_FMT_MXFP4) ? 6.0 : 2688.0;",
                       "const double R = 2688.0;"),
}


def mx_pins():
    failed = []
    for name, fn in (("group", test_mx_group_quantizer_bruteforce),
                     ("exact", lambda: test_mx_exactly_quantizable_inputs_reproduce_softmax(300, True)),
                     ("equal_k", lambda: test_mx_all_keys_equal_gives_mean_of_decoded_v(False))):
        try:
            fn()
        except Exception:
            failed.append(name)
    return failed


@pytest.mark.parametrize("name", sorted(MX_MUTATIONS))
def test_planted_mx_mistake_is_caught(name, tmp_path):
    old, new = MX_MUTATIONS[name]
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, name
    mutated = tmp_path / "sage_oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "sage_oracle.h").write_text(open(ORACLE_SRC[:-2] + ".h").read())
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    str(mutated), "-o", str(so), "-lm"], check=True)
    with oracle.swapped(str(so)):
        assert mx_pins(), f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_mx_pins():
    assert mx_pins() == []


def test_mx_format_matches_the_page():
    import json
    facts = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))
    mx = facts["mxfp4_group"]
    assert oracle.GROUP["mxfp4"] == mx["size"] == 32 and mx["scale_format"] == "E8M0"
    # an E8M0 scale is a pure power of two: 2^-127 .. 2^127, no mantissa
    vals = [oracle.e8m0_value(b) for b in range(255)]
    assert all(np.frexp(v)[0] == 0.5 for v in vals)
    assert vals[0] == 2.0 ** -127 and vals[254] == 2.0 ** 127
