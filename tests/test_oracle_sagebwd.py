"""Pins for the SageBwd oracle (oracle/sagebwd_oracle.c): 8-bit attention for
training, forward and backward (senqingzn.com article on SageAttention3,
"INT8 attention for training").

* the INT8 quantizer, by brute force: each code is the integer in
  [-127, 127] nearest to x * (127 / amax) (float arithmetic, ties to even),
  and a block's largest magnitude maps to +-127;
* the algebra, with every rounding step off: float64 softmax attention and
  its gradient from torch's float64 autograd, to 1e-10;
* the scales, by exact identities: Q -> 2Q at scale c equals Q at scale 2c
  (INT8 codes unchanged, scales doubled); V -> 2V doubles O, dQ and dK and
  leaves dV; dO -> 2 dO doubles the three gradients and leaves O;
* that the products use the quantized operands: a V block (or dO block) with
  one outlier quantizes every other entry of that block to zero, so channels
  without the outlier must come out exactly zero;
* FP16 rounding of dP's operands: a power-of-two scaling of dO scales every
  gradient exactly until dO reaches FP16's subnormal range, and dQ not after;
* the shape of the P and dS blocks (64 queries x 128 keys): query rows in
  different 64-row blocks never interact (changing rows 64-127 leaves O,
  lse, dQ of rows 0-63 and every dK, dV entry bit-identical when their dO
  rows are zero), while rows of one block share a scale (changing rows 32-63
  changes O of rows 0-31);
* planted mistakes, each caught by at least one of the above.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "sagebwd_oracle.c")


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def rand_inputs(BH, N, D, seed, scales=(1.0, 1.0, 1.0, 1.0)):
    rng = np.random.default_rng(seed)
    return [bf16(rng.standard_normal((BH, N, D)) * s) for s in scales]


def torch_reference(q, k, v, do, causal, scale):
    qf, kf, vf = (t.double().requires_grad_() for t in (q, k, v))
    s = torch.einsum("bid,bjd->bij", qf, kf) * scale
    if causal:
        N = s.shape[-1]
        s = s.masked_fill(~torch.tril(torch.ones(N, N, dtype=torch.bool)), float("-inf"))
    lse = torch.logsumexp(s, -1)
    o = torch.einsum("bij,bjd->bid", torch.softmax(s, -1), vf)
    o.backward(do.double())
    return o.detach().numpy(), lse.detach().numpy(), qf.grad.numpy(), kf.grad.numpy(), vf.grad.numpy()


def test_int8_code_is_the_nearest_integer_ties_even():
    rng = np.random.default_rng(1)
    amax = np.float32(3.7)
    inv = np.float32(127.0) / amax
    cands = np.arange(-127, 128, dtype=np.float64)
    xs = list(rng.uniform(-3.7, 3.7, 4000).astype(np.float32))
    # values landing on half-integers after the product, both signs
    xs += [np.float32(c + 0.5) / inv for c in range(-126, 126, 7)]
    for x in xs:
        y = np.float32(x) * inv  # one float product, rounded to nearest
        d = np.abs(cands - np.float64(y))
        best = cands[d == d.min()]
        want = best[0] if best.size == 1 else best[np.abs(best) % 2 == 0][0]
        assert oracle.int8_code(float(x), float(amax)) == int(want), (x, y)
    assert oracle.int8_code(3.7, 3.7) == 127 and oracle.int8_code(-3.7, 3.7) == -127
    assert oracle.int8_code(1.0, 0.0) == 0
    assert oracle.int8_scale(127.0) == 1.0


@pytest.mark.parametrize("N,D", [(1, 64), (130, 64), (300, 128)])
def test_block_quantizer(N, D):
    BH = 2
    (x,) = rand_inputs(BH, N, D, seed=N, scales=(2.0,))
    codes, scales = oracle.sagebwd_quantize(x, BH, N, D)
    xv = x.float().numpy()
    nb = (N + 127) // 128
    assert scales.shape == (BH, nb)
    for b in range(BH):
        for blk in range(nb):
            sl = slice(128 * blk, min(N, 128 * blk + 128))
            amax = np.abs(xv[b, sl]).max()
            assert scales[b, blk] == np.float32(amax) / np.float32(127)
            c = codes[b, sl].astype(np.int64)
            assert np.abs(c).max() == 127 and np.abs(c).max() <= 127
            # every code within half a step of x / s
            assert np.all(np.abs(xv[b, sl] / scales[b, blk] - c) <= 0.5 + 1e-5)


@pytest.mark.parametrize("N,D,causal", [(200, 64, False), (300, 64, True), (130, 128, True)])
def test_exact_mode_is_attention_and_its_gradient(N, D, causal):
    BH = 2
    q, k, v, do = rand_inputs(BH, N, D, seed=N + D, scales=(1.0, 1.5, 1.0, 1.0))
    scale = 1.0 / np.sqrt(D)
    got = oracle.sagebwd(q, k, v, do, BH, N, D, causal, scale, quant=False)
    want = torch_reference(q, k, v, do, causal, scale)
    for name, g, w in zip(("o", "lse", "dq", "dk", "dv"), got, want):
        assert np.abs(g - w).max() <= 1e-10 * max(1.0, np.abs(w).max()), name


@pytest.mark.parametrize("causal", [False, True])
def test_scale_identities(causal):
    BH, N, D = 2, 260, 64
    q, k, v, do = rand_inputs(BH, N, D, seed=5)
    two = lambda t: (t.float() * 2).to(torch.bfloat16)
    c = 0.11
    base = oracle.sagebwd(q, k, v, do, BH, N, D, causal, c)
    # 2Q at scale c == Q at scale 2c: same forward; dQ halves, dK equal
    a = oracle.sagebwd(two(q), k, v, do, BH, N, D, causal, c)
    b = oracle.sagebwd(q, k, v, do, BH, N, D, causal, 2 * c)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(a[2], b[2] / 2) and np.array_equal(a[3], b[3]) and np.array_equal(a[4], b[4])
    assert not np.array_equal(b[0], base[0])
    # 2V: O, dQ, dK double; dV unchanged
    o2, l2, dq2, dk2, dv2 = oracle.sagebwd(q, k, two(v), do, BH, N, D, causal, c)
    assert np.array_equal(o2, 2 * base[0]) and np.array_equal(l2, base[1])
    assert np.array_equal(dq2, 2 * base[2]) and np.array_equal(dk2, 2 * base[3])
    assert np.array_equal(dv2, base[4])
    # 2 dO: O unchanged, every gradient doubles
    o3, _, dq3, dk3, dv3 = oracle.sagebwd(q, k, v, two(do), BH, N, D, causal, c)
    assert np.array_equal(o3, base[0])
    assert np.array_equal(dq3, 2 * base[2]) and np.array_equal(dk3, 2 * base[3])
    assert np.array_equal(dv3, 2 * base[4])


def test_dp_operands_are_rounded_to_fp16():
    """Scaling dO by a power of two is exact for the INT8 blocks, D and bf16;
    only dP's FP16 operands break it, once dO falls into FP16's subnormal
    range (below 2^-14): dQ then stops scaling by exactly 2^-18."""
    BH, N, D = 2, 200, 64
    q, k, v, do = rand_inputs(BH, N, D, seed=7)
    small = (do.float() * 2.0 ** -18).to(torch.bfloat16)
    base = oracle.sagebwd(q, k, v, do, BH, N, D, False)
    tiny = oracle.sagebwd(q, k, v, small, BH, N, D, False)
    assert np.array_equal(tiny[4], base[4] * 2.0 ** -18)          # dV: INT8 dO only
    assert not np.array_equal(tiny[2], base[2] * 2.0 ** -18)      # dQ: through dP
    ex = oracle.sagebwd(q, k, v, do, BH, N, D, False, quant=False)
    ex_tiny = oracle.sagebwd(q, k, v, small, BH, N, D, False, quant=False)
    assert np.array_equal(ex_tiny[2], ex[2] * 2.0 ** -18)


def test_products_use_the_quantized_v_and_do():
    # Every V (and dO) entry is 1 except one outlier of 1000 in channel 0 of
    # token 0: per 128-token block the scale is 1000/127, so the 1s quantize
    # to code 0.  O and dV are then exactly zero in every channel but 0 (for
    # N <= 128: one block); without quantization they are not.
    BH, N, D = 1, 100, 64
    rng = np.random.default_rng(3)
    q, k = (bf16(rng.standard_normal((BH, N, D))) for _ in range(2))
    big = np.ones((BH, N, D), np.float32)
    big[0, 0, 0] = 1000.0
    v = do = bf16(big)
    o, _, _, _, dv = oracle.sagebwd(q, k, v, do, BH, N, D, False)
    # channel 0 holds P^[i, 0] * 1000; small P entries may quantize to 0 too
    assert np.all(o[0, :, 1:] == 0.0) and np.all(o[0, :, 0] >= 0) and np.any(o[0, :, 0] > 0)
    assert np.all(dv[0, :, 1:] == 0.0) and np.any(dv[0, :, 0] != 0)
    oe, _, _, _, dve = oracle.sagebwd(q, k, v, do, BH, N, D, False, quant=False)
    assert np.abs(oe[0, :, 1:] - 1.0).max() < 1e-12 and np.all(dve[0, :, 1:] != 0.0)


def block_case(changed_rows, zero_do_rows):
    """Two key tiles.  Every query row is aligned with key 0 (tile 0), so its
    tile-1 probabilities are about e^-3; the rows in `changed_rows` of the
    variant are aligned with key 128 instead (tile-1 maximum 1).  q[0, 2] = 8
    holds the first Q block's maximum in both.  dO rows `zero_do_rows` are 0."""
    BH, N, D = 1, 256, 64
    rng = np.random.default_rng(11)
    k = rng.standard_normal((BH, N, D)) * 0.5
    k[0, 0, 0] = 6.0
    k[0, 128, 1] = 6.0
    q = np.clip(rng.standard_normal((BH, N, D)) * 0.3, -1, 1)
    q[0, :, 0] = 4.0
    q[0, 0, 2] = 8.0
    qv = q.copy()
    qv[0, changed_rows, 0] = 0.0
    qv[0, changed_rows, 1] = 4.0
    v = rng.standard_normal((BH, N, D))
    do = rng.standard_normal((BH, N, D))
    do[0, zero_do_rows] = 0.0
    args = (BH, N, D, False, 0.125)
    base = oracle.sagebwd(bf16(q), bf16(k), bf16(v), bf16(do), *args)
    var = oracle.sagebwd(bf16(qv), bf16(k), bf16(v), bf16(do), *args)
    return base, var


def test_p_blocks_are_64_queries_by_128_keys():
    rows = slice(64, 128)
    (o, lse, dq, dk, dv), (o2, lse2, dq2, dk2, dv2) = block_case(rows, rows)
    assert np.array_equal(o[0, :64], o2[0, :64]) and np.array_equal(lse[0, :64], lse2[0, :64])
    assert np.array_equal(dq[0, :64], dq2[0, :64])
    assert np.array_equal(dk, dk2) and np.array_equal(dv, dv2)
    assert not np.array_equal(o[0, 64:128], o2[0, 64:128])
    # within one block the scale is shared: rows 32-63 move rows 0-31
    rows = slice(32, 64)
    (o, *_), (o2, *_) = block_case(rows, rows)
    assert not np.array_equal(o[0, :32], o2[0, :32])


@pytest.mark.parametrize("N,D,causal", [(256, 64, False), (300, 128, True)])
def test_quantized_against_exact(N, D, causal):
    # measured (seed 6, k x1.5): cosine O >= 0.9996, dQ/dK/dV >= 0.9978; bound with headroom
    BH = 2
    q, k, v, do = rand_inputs(BH, N, D, seed=6, scales=(1.0, 1.5, 1.0, 1.0))
    qq = oracle.sagebwd(q, k, v, do, BH, N, D, causal)
    ex = oracle.sagebwd(q, k, v, do, BH, N, D, causal, quant=False)
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), qq, ex):
        cos = (a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum())
        print(name, cos)
        assert cos > 0.99, (name, cos)
        assert not np.array_equal(a, b) or name == "lse"


# ---------------------------------------------------------------- mutations
MUTATIONS = {
    "ds_sign": ("S[(size_t)i * N + j] = P[(size_t)i * N + j] * (dp - Dr[i]);",
                "S[(size_t)i * N + j] = P[(size_t)i * N + j] * (Dr[i] - dp);"),
    "ds_drops_D": ("S[(size_t)i * N + j] = P[(size_t)i * N + j] * (dp - Dr[i]);",
                   "S[(size_t)i * N + j] = P[(size_t)i * N + j] * dp;"),
    "dq_without_scale": ("dq[(size_t)i * D + d] = scale * acc[d];", "dq[(size_t)i * D + d] = acc[d];"),
    "dk_not_transposed": ("mt_times(Pq, Qd, N, D, dk);", "mt_times(Pq, Kd, N, D, dk);"),
    "dv_from_v": ("mt_times(Pq, dOd, N, D, dv);", "mt_times(Pq, Vd, N, D, dv);"),
    "mt_not_transposed": ("dst[(size_t)j * D + d] += M[(size_t)i * N + j] * X[(size_t)i * D + d];",
                          "dst[(size_t)j * D + d] += M[(size_t)j * N + i] * X[(size_t)i * D + d];"),
    "o_from_unquantized_v": ("dequant_head(v, N, D, quant, Vd);", "dequant_head(v, N, D, 0, Vd);"),
    "dv_from_unquantized_do": ("dequant_head(dout, N, D, quant, dOd);", "dequant_head(dout, N, D, 0, dOd);"),
    "lse_without_max": ("L[i] = m[i] + log(l[i]);", "L[i] = log(l[i]);"),
    "o_not_rescaled": ("for (int d = 0; d < D; d++) O[(size_t)i * D + d] *= alpha;", ""),
    "dp_unrounded_operands": ("dOh[x] = quant ? fp16_round(a) : (double)a;", "dOh[x] = (double)a;"),
    "l_not_rescaled": ("l[i] = l[i] * alpha + rs;", "l[i] = l[i] + rs;"),
    "p_block_128_queries": ("#define QBLK 64", "#define QBLK 128"),
    "p_block_one_row": ("#define QBLK 64", "#define QBLK 1"),
    "int8_ties_up": ("float c = rintf(y);", "float c = roundf(y);"),
}


def all_pins():
    checks = [
        ("code", test_int8_code_is_the_nearest_integer_ties_even),
        ("exact", lambda: test_exact_mode_is_attention_and_its_gradient(200, 64, False)),
        ("exact_causal", lambda: test_exact_mode_is_attention_and_its_gradient(130, 128, True)),
        ("scales", lambda: test_scale_identities(False)),
        ("outliers", test_products_use_the_quantized_v_and_do),
        ("blocks", test_p_blocks_are_64_queries_by_128_keys),
        ("fp16", test_dp_operands_are_rounded_to_fp16),
    ]
    failed = []
    for name, fn in checks:
        try:
            fn()
        except Exception:
            failed.append(name)
    return failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    d = os.path.dirname(SRC)
    (tmp_path / "sagebwd_oracle.c").write_text(src.replace(old, new))
    for f in ("sagebwd_oracle.h", "sage_oracle.c", "sage_oracle.h"):
        (tmp_path / f).write_text(open(os.path.join(d, f)).read())
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    str(tmp_path / "sage_oracle.c"), str(tmp_path / "sagebwd_oracle.c"), "-o", str(so), "-lm"],
                   check=True)
    sys.path.insert(0, os.path.dirname(__file__))
    with oracle.swapped(str(so)):
        failed = all_pins()
    assert failed, f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_all_pins():
    assert all_pins() == []
