"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/sage_fp4.h declares, sizes its workspace, and rejects
bad arguments before touching the device."""
import ctypes

import pytest

from bit_attention_gb300 import sage_fp4 as S


def test_library_exports_every_header_function():
    lib = S.load()
    names = S.header_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_bytes():
    # per (b,h): Q,K codes N_pad*D/2 and scales N_pad*D/16; V^T codes D*N_pad/2,
    # scales 128*N_pad/16; each part 256-aligned, plus 256 bytes of status
    B, H, N, D = 4, 32, 4096, 128
    BH, Np = B * H, 4096
    parts = [BH * Np * D // 2, BH * Np * D // 16] * 2 + [BH * D * Np // 2, BH * 128 * Np // 16]
    assert S.sage_fp4_workspace_bytes(B, H, N, D) == sum((p + 255) // 256 * 256 for p in parts) + 256
    assert S.sage_fp4_workspace_bytes(1, 1, 17, 64) > 0
    assert S.sage_fp4_workspace_bytes(1, 1, 17, 96) == 0
    assert S.sage_fp4_workspace_bytes(-1, 1, 17, 64) == 0


def test_workspace_carving_is_pointer_arithmetic():
    base = 0x7000_0000
    nbytes = S.sage_fp4_workspace_bytes(2, 3, 300, 64)
    rc, q = S.sage_fp4_qkv_from_workspace(base, nbytes, 2, 3, 300, 64)
    assert rc == 0
    ptrs = [q.q.codes, q.q.scales, q.k.codes, q.k.scales, q.vt.codes, q.vt.scales, q.status]
    assert ptrs == sorted(ptrs) and ptrs[0] == base
    assert all(p % 256 == 0 for p in ptrs)
    assert q.status + 4 <= base + nbytes
    assert S.sage_fp4_qkv_from_workspace(base, nbytes - 1, 2, 3, 300, 64)[0] == S.EINVAL
    assert S.sage_fp4_qkv_from_workspace(base + 16, nbytes, 2, 3, 300, 64)[0] == S.EINVAL


def _qkv():
    rc, q = S.sage_fp4_qkv_from_workspace(0x7000_0000, 1 << 30, 1, 2, 512, 128)
    assert rc == 0
    return q


@pytest.mark.parametrize("args", [
    dict(D=96), dict(N=-1), dict(B=-2), dict(o=0), dict(o=0x1008), dict(causal=2),
])
def test_attn_rejects_bad_arguments(args):
    a = dict(B=1, H=2, N=512, D=128, o=0x1000, causal=0)
    a.update(args)
    rc = S.sage_fp4_attn_fwd(_qkv(), a["o"], a["B"], a["H"], a["N"], a["D"], a["causal"], None)
    assert rc == S.EINVAL


def test_attn_rejects_bad_operands():
    q = _qkv()
    q.k.codes = 0
    assert S.sage_fp4_attn_fwd(q, 0x1000, 1, 2, 512, 128, 0, None) == S.EINVAL
    q = _qkv()
    q.vt.scales += 8
    assert S.sage_fp4_attn_fwd(q, 0x1000, 1, 2, 512, 128, 0, None) == S.EINVAL
    q = _qkv()
    q.status = 0
    assert S.sage_fp4_attn_fwd(q, 0x1000, 1, 2, 512, 128, 0, None) == S.EINVAL


def test_quantize_rejects_bad_arguments():
    q = _qkv()
    assert S.sage_fp4_quantize_qkv(0, 0x2000, 0x3000, q, 1, 2, 512, 128, None) == S.EINVAL
    assert S.sage_fp4_quantize_qkv(0x1004, 0x2000, 0x3000, q, 1, 2, 512, 128, None) == S.EINVAL
    assert S.sage_fp4_quantize_qkv(0x1000, 0x2000, 0x3000, q, 1, 2, 512, 80, None) == S.EINVAL


def test_empty_problems_are_no_ops():
    # nothing to compute: OK without touching the device
    q = _qkv()
    assert S.sage_fp4_attn_fwd(q, 0x1000, 0, 2, 512, 128, 0, None) == S.OK
    assert S.sage_fp4_attn_fwd(q, 0x1000, 1, 2, 0, 128, 1, None) == S.OK
    assert S.sage_fp4_quantize_qkv(0x1000, 0x2000, 0x3000, q, 1, 0, 512, 64, None) == S.OK


def test_probe_argument_checks():
    assert S.sage_fp4_mma_probe(0x1000, 0x2000, 0x3000, 0x4000, 96, 64, 0, 0x5000, 0x6000, None) == S.EINVAL
    assert S.sage_fp4_mma_probe(0x1000, 0x2000, 0x3000, 0x4000, 64, 32, 0, 0x5000, 0x6000, None) == S.EINVAL
    assert S.sage_fp4_cvt_probe(0, 16, None, None, None) == S.EINVAL
    # unknown option bits
    assert S.sage_fp4_mma_probe_ex(0x1000, 0x2000, 0x3000, 0x4000, 64, 64, 8, 0x5000, 0x6000, None) == S.EINVAL


def test_strerror():
    for code in (S.OK, S.EINVAL, S.ECUDA, S.ETIMEOUT, S.EUNSUPPORTED):
        assert S.strerror(code) and S.strerror(code) != "unknown status"
    assert S.strerror(12345) == "unknown status"


def test_host_workspace_bytes():
    # three slots, each: staged q, k, v, o of c = ceil(B*H/8) heads (256-aligned)
    # plus the quantized operands of c heads
    B, H, N, D = 4, 32, 4096, 128
    c = -(-B * H // 8)
    stage = (c * N * D * 2 + 255) // 256 * 256
    qws = (S.sage_fp4_workspace_bytes(1, c, N, D) + 255) // 256 * 256
    assert S.sage_fp4_host_workspace_bytes(B, H, N, D) == 3 * (4 * stage + qws)
    # fewer heads than chunks: one head per chunk
    c1 = (300 * 64 * 2 + 255) // 256 * 256
    assert S.sage_fp4_host_workspace_bytes(1, 3, 300, 64) == 3 * (4 * c1 + S.sage_fp4_workspace_bytes(1, 1, 300, 64))
    assert S.sage_fp4_host_workspace_bytes(1, 1, 17, 96) == 0
    assert S.sage_fp4_host_workspace_bytes(-1, 1, 17, 64) == 0
    assert S.sage_fp4_host_workspace_bytes(0, 4, 17, 64) == 256


def test_host_pipeline_rejects_bad_arguments():
    B, H, N, D = 1, 2, 512, 128
    ws = S.sage_fp4_host_workspace_bytes(B, H, N, D)
    good = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, B=B, H=H, N=N, D=D, causal=0,
                ws=0x7000_0000, nbytes=ws, status=0x5000)

    def call(**kw):
        a = dict(good)
        a.update(kw)
        return S.sage_fp4_attention_host(a["q"], a["k"], a["v"], a["o"], a["B"], a["H"], a["N"],
                                         a["D"], a["causal"], a["ws"], a["nbytes"], a["status"], None)

    for bad in (dict(q=0), dict(o=0), dict(status=0), dict(status=0x5002), dict(ws=0),
                dict(ws=0x7000_0010), dict(nbytes=ws - 1), dict(causal=2), dict(D=96), dict(N=-1)):
        assert call(**bad) == S.EINVAL, bad
    # nothing to compute: OK without touching the device
    assert call(B=0) == S.OK
    assert call(N=0, nbytes=256) == S.OK


def test_strided_quantize_and_scaled_attention_reject_bad_arguments():
    q = _qkv()
    B, H, N, D = 1, 2, 512, 128

    def quant(sq=None, sk=None, sv=None, fmt=0):
        return S.sage_fp4_quantize_qkv_strided(0x1000, sq, 0x2000, sk, 0x3000, sv, q, B, H, N, D, None, fmt)

    nhd = S.sage_fp4_strides(N * H * D, D, H * D)
    for bad in (S.sage_fp4_strides(N * H * D, D, H * D + 4),   # 8-byte rows
                S.sage_fp4_strides(-8, D, H * D),               # negative
                S.sage_fp4_strides(N * H * D, 1 << 62, H * D)):  # offsets past 2^62
        assert quant(sq=bad) == S.EINVAL
        assert quant(sv=bad) == S.EINVAL
    assert quant(fmt=3) == S.EINVAL and quant(fmt=-1) == S.EINVAL
    assert S.sage_fp4_quantize_qkv_strided(0x1000, nhd, 0x2000, nhd, 0x3000, nhd, q, 0, H, N, D, None) == S.OK

    def attn(scale, so=None, causal=0, fmt=0):
        return S.sage_fp4_attn_fwd_ex(q, 0x4000, so, B, H, N, D, causal, scale, None, fmt)

    for bad in (0.0, -0.1, float("inf"), float("nan"), 1e31):
        assert attn(bad) == S.EINVAL, bad
    assert attn(0.1, so=S.sage_fp4_strides(N * H * D, D, 12)) == S.EINVAL
    assert attn(0.1, fmt=7) == S.EINVAL
    assert S.sage_fp4_attn_fwd_ex(q, 0x4000, nhd, 0, H, N, D, 0, 0.1, None) == S.OK


def test_torch_op_is_registered_with_a_fake():
    import torch
    from torch._subclasses.fake_tensor import FakeTensorMode
    import bit_attention_gb300.torch_op  # noqa: F401  (registers the op)
    with FakeTensorMode():
        x = torch.empty(2, 300, 3, 64, dtype=torch.bfloat16)
        o = torch.ops.sage_fp4.attention(x, x, x, True, 0.2, "NHD")
        assert o.shape == x.shape and o.dtype == torch.bfloat16 and o.is_contiguous()


def test_binding_argument_counts_match_the_header():
    import re
    text = open(S._HEADER).read()
    decls = dict(re.findall(r"^(?:int|size_t|const char \*)\s*(sage_fp4_\w+)\(([^;]*)\);", text, re.M))
    lib = S.load()
    assert set(decls) == set(S.header_functions())
    for name, args in decls.items():
        n = len([a for a in args.replace("\n", " ").split(",") if a.strip() and a.strip() != "void"])
        assert len(getattr(lib, name).argtypes) == n, name


def test_noalloc_rejects_before_touching_the_device():
    # sizes are checked first (EINVAL for invalid ones, ETOOLARGE above the
    # fixed scratch array), then pointers; none of these reaches the device
    f = S.sage_fp4_attention_noalloc
    good = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000)
    assert f(*good, 1, 2, 512, 96, 0, None) == S.EINVAL
    assert f(*good, -1, 2, 512, 128, 0, None) == S.EINVAL
    assert f(*good, 1, 2, 512, 128, 2, None) == S.EINVAL
    assert f(*good, 4, 32, 4096, 128, 0, None) == S.ETOOLARGE
    assert f(0x1008, *good[1:], 1, 2, 512, 128, 0, None) == S.EINVAL
    assert f(*good[:4], 0x5002, 1, 2, 512, 128, 0, None) == S.EINVAL
    assert f(*good[:4], 0, 1, 2, 512, 128, 0, None) == S.EINVAL
    assert f(*good, 0, 2, 512, 128, 0, None) == S.OK  # empty: a no-op


def test_directp_format_takes_contiguous_o_only():
    # SAGE_FP4_FORMAT_MXFP4_DIRECTP (2) with O through other strides is
    # refused before anything touches the device; a format past it is too
    q = _qkv()
    nhd = S.sage_fp4_strides(512 * 2 * 128, 128, 2 * 128)  # [B,N,H,D] strides of B1 H2 N512 D128
    assert S.sage_fp4_attn_fwd_ex(q, 0x1000, nhd, 1, 2, 512, 128, 0, 0.1, None, 2) == S.EINVAL
    assert S.sage_fp4_attn_fwd_ex(q, 0x1000, None, 1, 2, 512, 128, 0, 0.1, None, 3) == S.EINVAL


def test_debug_build_loads_and_exports_every_header_function():
    # the bounds-checking build of the same sources (SAGE_FP4_DEBUG_BOUNDS=1)
    lib = S.load(debug_bounds=True)
    for n in S.header_functions():
        assert hasattr(lib, n), n
    assert lib is not S.load()
    assert "debug build" in S.load(debug_bounds=True).sage_fp4_strerror(S.EBOUNDS).decode()
