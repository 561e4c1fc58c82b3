"""The MXFP4 variant on the GPU (1x32 groups, E8M0 scales).

[NEWS-HW] weighs MXFP4 against NVFP4 and keeps NVFP4; this variant swaps the
microscaling format in every quantization step (Q, K, V and P) and runs the
products on `kind::mxf4` tensor cores.  Checked against the oracle's MXFP4
variant:

* the tensor-core product (`sage_fp4_mma_probe_mx`) equals the exact product
  of the decoded operands, with bytes 2-3 of every scale word filled with
  noise that must not be read;
* the quantized operands are bit-exact, including a strided (NHD) input;
* attention O is within the attention tests' tolerance of the oracle, on
  small shapes in full and on the LLM workload on sampled rows;
* at full size, NVFP4 is more accurate than MXFP4 against exact attention on
  every workload pattern, the pages' finding.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300.synth import WORKLOADS, make_qkv
from helpers import block_offsets, check_o, cosine, rel_l1, sample_rows

pytestmark = pytest.mark.gpu

E2M1 = np.array([oracle.e2m1_value(c) for c in range(16)])


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _mx_block(plain32, rng=None):
    """[R, C/32] E8M0 bytes -> block layout: bytes 0-1 of each step's word; bytes 2-3
    zero (or noise when rng is given)."""
    R, g32 = plain32.shape
    g16 = 2 * g32
    out = np.zeros(R * g16, np.uint8)
    if rng is not None:
        out[:] = rng.integers(0, 256, size=out.size, dtype=np.uint8)
    off = block_offsets(R, g16)
    for g in range(g32):
        out[off[:, 4 * (g // 2) + g % 2]] = plain32[:, g]
        if rng is None:
            out[off[:, 4 * (g // 2) + 2 + g % 2]] = 0
    return out


def _mx_plain(block, R, C):
    """Block-layout MX scales [.., R*C/16] -> ([.., R, C/32] E8M0 bytes, padding bytes)."""
    g16 = C // 16
    off = block_offsets(R, g16)
    blk = block.reshape(*block.shape[:-1], R * g16)
    plain = np.stack([blk[..., off[:, 4 * (g // 2) + g % 2]] for g in range(C // 32)], axis=-1)
    pad = np.stack([blk[..., off[:, 4 * (g // 2) + 2 + g % 2]] for g in range(C // 32)], axis=-1)
    return plain, pad


@pytest.mark.parametrize("K", [64, 128, 256])
@pytest.mark.parametrize("n", [64, 128])
@pytest.mark.parametrize("a_by_threads", [0, 1])
@pytest.mark.parametrize("sf_rows128", [0, 1])
def test_mx_mma_probe_exact_product(K, n, a_by_threads, sf_rows128):
    rng = np.random.default_rng(K * 3 + n + a_by_threads)

    def operand(rows):
        codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
        sc = np.zeros((128, K // 32), np.uint8)
        sc[:rows] = rng.integers(120, 135, size=(rows, K // 32), dtype=np.uint8)  # 2^-7 .. 2^7
        dec = E2M1[codes] * np.repeat(2.0 ** (sc[:rows].astype(np.float64) - 127), 32, axis=1)
        return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), _mx_block(sc, rng), dec

    (ac, asf, ad), (bc, bsf, bd) = operand(128), operand(n)
    ta, tsa, tb, tsb = _dev(ac), _dev(asf), _dev(bc), _dev(bsf)
    d = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = S.PROBE_MX | (S.PROBE_A_BY_THREADS if a_by_threads else 0) | (S.PROBE_SF_ROWS128 if sf_rows128 else 0)
    rc = S.sage_fp4_mma_probe_ex(ta.data_ptr(), tsa.data_ptr(), tb.data_ptr(), tsb.data_ptr(), n, K,
                                 flags, d.data_ptr(), status.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = d.cpu().numpy().astype(np.float64)
    err = np.abs(got - ad @ bd.T) / np.maximum(np.abs(ad) @ np.abs(bd).T, 1e-30)
    assert np.isfinite(got).all() and err.max() < 1e-5, err.max()


@pytest.mark.parametrize("B,H,N,D,pattern,nhd", [
    (1, 2, 300, 128, "iid", False),
    (2, 3, 333, 64, "k_channel_outliers", False),
    (1, 1, 17, 128, "sparse_outliers", False),
    (2, 2, 200, 128, "k_head_mean", True),
])
def test_mx_quantization_is_bit_exact(B, H, N, D, pattern, nhd):
    q, k, v = make_qkv(B, H, N, D, pattern, seed=N + D)
    BH, Np = B * H, oracle.round_up(N, 128)
    if nhd:
        qn, kn, vn = (x.transpose(1, 2).contiguous().cuda() for x in (q, k, v))
        z = S.QuantizedQKV(B, H, N, D)
        st = [S._bhnd(x, "NHD", "x")[1] for x in (qn, kn, vn)]
        assert S.sage_fp4_quantize_qkv_strided(qn.data_ptr(), st[0], kn.data_ptr(), st[1], vn.data_ptr(),
                                               st[2], z.struct, B, H, N, D,
                                               torch.cuda.current_stream().cuda_stream, 1) == S.OK
    else:
        z = S.quantize_qkv(q.cuda(), k.cuda(), v.cuda(), fmt="mxfp4")
    torch.cuda.synchronize()
    assert z.get_status() == 0
    ref = oracle.Quantized(q, k, v, BH, N, D, fmt="mxfp4")
    assert np.array_equal(z.q_codes.cpu().numpy(), ref.qc)
    assert np.array_equal(z.k_codes.cpu().numpy(), ref.kc)
    assert np.array_equal(z.vt_codes.cpu().numpy(), ref.vc)
    for got, want, R, C in ((z.q_scales, ref.qs, Np, D), (z.k_scales, ref.ks, Np, D),
                            (z.vt_scales, ref.vs, 128, Np)):
        plain, pad = _mx_plain(got.cpu().numpy(), R, C)
        assert not pad.any()
        rows = want.shape[1]
        assert np.array_equal(plain[:, :rows], want)


def _mx_attention(q, k, v, causal):
    z = S.quantize_qkv(q.cuda(), k.cuda(), v.cuda(), fmt="mxfp4")
    o = S.attn_fwd(z, causal, out=torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert z.get_status() == 0
    return o


@pytest.mark.parametrize("B,H,N,D,causal,pattern", [
    (1, 2, 512, 128, False, "iid"),
    (1, 2, 300, 128, True, "k_channel_outliers"),
    (2, 2, 300, 64, False, "k_head_mean"),
    (1, 1, 17, 64, True, "iid"),
    (1, 2, 1100, 128, False, "sparse_outliers"),
])
def test_mx_attention_matches_oracle(B, H, N, D, causal, pattern):
    q, k, v = make_qkv(B, H, N, D, pattern, seed=31 + N)
    got = _mx_attention(q, k, v, causal).float().cpu().numpy().reshape(B * H * N, D)
    ref = oracle.attention(oracle.Quantized(q, k, v, B * H, N, D, fmt="mxfp4"), causal)[0]
    check_o(got, ref, f"mx B{B} H{H} N{N} D{D} causal={causal} {pattern}")


def _mx_fuzz_cases(n=6, seed=77):
    rng = np.random.default_rng(seed)
    pats = ["iid", "k_channel_outliers", "k_head_mean", "sparse_outliers"]
    return [(int(rng.integers(1, 3)), int(rng.integers(1, 3)), int(rng.integers(1, 600)),
             int(rng.choice([64, 128])), bool(rng.integers(0, 2)), pats[int(rng.integers(0, 4))])
            for _ in range(n)]


@pytest.mark.parametrize("B,H,N,D,causal,pattern", _mx_fuzz_cases())
def test_mx_attention_random_shapes(B, H, N, D, causal, pattern):
    q, k, v = make_qkv(B, H, N, D, pattern, seed=5 * N + D)
    got = _mx_attention(q, k, v, causal).float().cpu().numpy().reshape(B * H * N, D)
    ref = oracle.attention(oracle.Quantized(q, k, v, B * H, N, D, fmt="mxfp4"), causal)[0]
    check_o(got, ref, f"mx fuzz B{B} H{H} N{N} D{D} causal={causal} {pattern}")


def test_mx_attention_llm_workload_sampled_rows():
    w = WORKLOADS["llm"]
    q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.pattern, seed=0)
    got = _mx_attention(q, k, v, w.causal).float().cpu().numpy().reshape(-1, w.D)
    rows = sample_rows(w.B * w.H, w.N, per_head=4)
    ref = oracle.attention(oracle.Quantized(q, k, v, w.B * w.H, w.N, w.D, fmt="mxfp4"), w.causal,
                           rows=rows)[0]
    assert np.isfinite(got).all()
    check_o(got[rows], ref, "mx llm sampled rows")


@pytest.mark.parametrize("name", ["llm", "dit", "dit_long"])
def test_nvfp4_beats_mxfp4_at_full_size(name):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.pattern, seed=0)
    rows = np.sort(np.random.default_rng(1).choice(w.B * w.H * w.N, size=256, replace=False))
    exact = oracle.attention_exact(q, k, v, w.B * w.H, w.N, w.D, w.causal, rows=rows)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    res = {}
    for fmt in ("nvfp4", "mxfp4", "mxfp4_directp"):
        o = S.attn_fwd(S.quantize_qkv(qd, kd, vd, fmt=fmt), w.causal)
        got = o.float().cpu().numpy().reshape(-1, w.D)[rows]
        res[fmt] = (cosine(got, exact), rel_l1(got, exact))
    print(name, {f: tuple(round(x, 4) for x in r) for f, r in res.items()})
    assert res["nvfp4"][0] > res["mxfp4"][0] and res["nvfp4"][1] < res["mxfp4"][1], res


@pytest.mark.parametrize("D,causal", [(128, False), (64, True)])
def test_mx_strided_layout_matches_contiguous(D, causal):
    # the MXFP4 instantiation that writes O through strides (NHD), against the
    # dense one: the same bits
    B, H, N = 2, 3, 333
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "k_channel_outliers", seed=D + 7))
    want = S.attention(q, k, v, causal, fmt="mxfp4")
    qn, kn, vn = (x.transpose(1, 2).contiguous() for x in (q, k, v))
    got = S.attention(qn, kn, vn, causal, layout="NHD", fmt="mxfp4")
    torch.cuda.synchronize()
    assert torch.equal(got.transpose(1, 2), want)


# ------------------------------------------------------------------ Direct-P
def _dp_attention(q, k, v, causal):
    z = S.quantize_qkv(q.cuda(), k.cuda(), v.cuda(), fmt="mxfp4_directp")
    o = S.attn_fwd(z, causal, out=torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert z.get_status() == 0
    return o


@pytest.mark.parametrize("B,H,N,D,causal,pattern", [
    (1, 2, 512, 128, False, "iid"),
    (1, 2, 300, 128, True, "k_channel_outliers"),
    (2, 2, 300, 64, False, "k_head_mean"),
    (1, 1, 17, 64, True, "iid"),
    (1, 2, 1100, 128, False, "sparse_outliers"),
])
def test_directp_attention_matches_oracle(B, H, N, D, causal, pattern):
    # Direct-P: MXFP4 with l summed from the rounded P, against the oracle's
    # rounded normaliser (same tolerance and row checks as every attention test)
    q, k, v = make_qkv(B, H, N, D, pattern, seed=41 + N)
    got = _dp_attention(q, k, v, causal).float().cpu().numpy().reshape(B * H * N, D)
    qz = oracle.Quantized(q, k, v, B * H, N, D, fmt="mxfp4")
    ref = oracle.attention(qz, causal, lnorm="rounded")[0]
    check_o(got, ref, f"directp B{B} H{H} N{N} D{D} causal={causal} {pattern}")


def test_directp_llm_workload_sampled_rows():
    w = WORKLOADS["llm"]
    q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.pattern, seed=0)
    got = _dp_attention(q, k, v, w.causal).float().cpu().numpy().reshape(-1, w.D)
    rows = sample_rows(w.B * w.H, w.N, per_head=4)
    qz = oracle.Quantized(q, k, v, w.B * w.H, w.N, w.D, fmt="mxfp4")
    ref = oracle.attention(qz, w.causal, rows=rows, lnorm="rounded")[0]
    assert np.isfinite(got).all()
    check_o(got[rows], ref, "directp llm sampled rows")


@pytest.mark.parametrize("D,causal", [(128, False), (64, True)])
def test_directp_constant_v_is_returned(D, causal):
    # l and PV sum the same rounded P, so V = 1.5 everywhere gives O = 1.5
    # up to the FP32 sums' order and the bf16 rounding of O
    B, H, N = 1, 2, 700
    q, k, _ = make_qkv(B, H, N, D, "k_channel_outliers", seed=D)
    v = torch.full((B, H, N, D), 1.5, dtype=torch.bfloat16)
    o = _dp_attention(q, k, v, causal).float()
    assert (o - 1.5).abs().max().item() <= 2 ** -8 * 1.5
