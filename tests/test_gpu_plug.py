"""The plug-and-play attention: any layout with a contiguous D axis, an
explicit softmax scale, and the torch custom op.

Layouts and strides change only where the kernels read and write, never what
they compute, so every strided result must equal the contiguous [B,H,N,D]
one bit for bit: NHD tensors, Q/K/V viewed out of a packed [B,N,3,H,D]
tensor (each tile copied token row by token row), a slice along N, and the
quantized operands themselves.  A non-default softmax scale is compared
with the oracle at that scale (same tolerance as the attention tests).
"""
import pytest
import torch

import oracle
from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300.synth import make_qkv
from helpers import check_o

pytestmark = pytest.mark.gpu


def _cuda(*ts):
    return [t.cuda() for t in ts]


@pytest.mark.parametrize("B,H,N,D,causal", [(2, 3, 300, 128, False), (1, 4, 700, 64, True)])
def test_nhd_and_packed_views_match_contiguous(B, H, N, D, causal):
    q, k, v = _cuda(*make_qkv(B, H, N, D, "k_channel_outliers", seed=N + D))
    want = S.attention(q, k, v, causal)
    # NHD copies
    qn, kn, vn = (x.transpose(1, 2).contiguous() for x in (q, k, v))
    o_nhd = S.attention(qn, kn, vn, causal, layout="NHD")
    assert o_nhd.shape == (B, N, H, D)
    assert torch.equal(o_nhd.transpose(1, 2), want)
    # views into one packed [B, N, 3, H, D] tensor: token stride 3*H*D
    packed = torch.stack([qn, kn, vn], dim=2)
    o_packed = S.attention(packed[:, :, 0], packed[:, :, 1], packed[:, :, 2], causal, layout="NHD")
    assert torch.equal(o_packed, o_nhd)
    # HND slices of longer sequences, O written into a strided view
    big = [torch.cat([x, torch.randn_like(x[:, :, :40])], dim=2) for x in (q, k, v)]
    out_big = torch.zeros(B, H, N + 24, D, dtype=torch.bfloat16, device="cuda")
    S.attention(*(x[:, :, :N] for x in big), causal, out=out_big[:, :, 24:])
    torch.cuda.synchronize()
    assert torch.equal(out_big[:, :, 24:], want)
    assert not out_big[:, :, :24].any()


def test_strided_quantization_is_bit_identical():
    B, H, N, D = 2, 3, 333, 128
    q, k, v = _cuda(*make_qkv(B, H, N, D, "iid", seed=3))
    ref = S.quantize_qkv(q, k, v)
    packed = torch.stack([x.transpose(1, 2) for x in (q, k, v)], dim=2)  # [B,N,3,H,D]
    z = S.QuantizedQKV(B, H, N, D)
    st = [S._bhnd(packed[:, :, i], "NHD", "x")[1] for i in range(3)]
    rc = S.sage_fp4_quantize_qkv_strided(packed[:, :, 0].data_ptr(), st[0], packed[:, :, 1].data_ptr(), st[1],
                                         packed[:, :, 2].data_ptr(), st[2], z.struct, B, H, N, D,
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == S.OK
    torch.cuda.synchronize()
    assert z.get_status() == 0
    for part in ("q_codes", "q_scales", "k_codes", "k_scales", "vt_codes", "vt_scales"):
        assert torch.equal(getattr(z, part), getattr(ref, part)), part


@pytest.mark.parametrize("B,H,N,D,causal,scale", [
    (1, 2, 300, 128, True, 0.04),
    (2, 2, 500, 64, False, 0.3),
])
def test_softmax_scale_matches_oracle(B, H, N, D, causal, scale):
    q, k, v = make_qkv(B, H, N, D, "iid", seed=21)
    o = S.attention(*_cuda(q, k, v), causal, scale=scale)
    got = o.float().cpu().numpy().reshape(B * H * N, D)
    ref = oracle.attention(oracle.Quantized(q, k, v, B * H, N, D), causal, scale=scale)[0]
    check_o(got, ref, f"scale {scale} B{B} H{H} N{N} D{D} causal={causal}")
    # the default scale is 1/sqrt(D), and a different scale changes the result
    assert torch.equal(S.attention(*_cuda(q, k, v), causal, scale=1 / D ** 0.5),
                       S.attention(*_cuda(q, k, v), causal))
    assert not torch.equal(o, S.attention(*_cuda(q, k, v), causal))


def test_torch_custom_op_eager_and_compiled():
    import bit_attention_gb300.torch_op  # noqa: F401  (registers torch.ops.sage_fp4.attention)
    B, H, N, D = 1, 4, 384, 64
    qn, kn, vn = (x.transpose(1, 2).contiguous() for x in _cuda(*make_qkv(B, H, N, D, "iid", seed=8)))
    want = S.attention(qn, kn, vn, True, scale=0.2, layout="NHD")
    got = torch.ops.sage_fp4.attention(qn, kn, vn, True, 0.2, "NHD")
    assert torch.equal(got, want)

    def f(a, b, c):
        return torch.ops.sage_fp4.attention(a, b, c, True, 0.2, "NHD") * 2

    compiled = torch.compile(f, backend="eager", fullgraph=True)
    assert torch.equal(compiled(qn, kn, vn), want * 2)
