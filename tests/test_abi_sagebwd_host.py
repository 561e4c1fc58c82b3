"""Host-side checks of the SageBwd C ABI (include/sagebwd.h) that need no
GPU: every declared function is exported with the argument count the header
gives, the workspace layout is consistent, and bad arguments are rejected
before anything touches the device."""
import re

from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300 import sagebwd as SB


def test_library_exports_every_header_function():
    lib = SB.lib()
    names = SB.header_functions()
    assert len(names) == 16
    text = open(SB._HEADER).read()
    decls = dict(re.findall(r"^(?:int|size_t)\s*(sagebwd_\w+)\(([^;]*)\);", text, re.M))
    assert set(decls) == set(names)
    for name, args in decls.items():
        n = len([a for a in args.replace("\n", " ").split(",") if a.strip()])
        assert len(getattr(lib, name).argtypes) == n, name


def test_workspace_layout():
    B, H, N, D = 2, 3, 300, 64
    BH, Np = B * H, 384
    rc, offs = SB.sagebwd_workspace_layout(B, H, N, D)
    assert rc == S.OK and len(offs) == SB.WS_FIELDS
    total = SB.sagebwd_workspace_bytes(B, H, N, D)
    sizes = [2 * BH * Np * D] * 9 + [4 * BH * 3] * 4 + [4 * BH * Np] * 2 + [4 * BH * Np * D, 256]
    assert offs[0] == 0
    for i, sz in enumerate(sizes):
        assert offs[i] % 256 == 0
        end = offs[i + 1] if i + 1 < len(offs) else total
        assert end - offs[i] == (sz + 255) // 256 * 256, SB.WS_NAMES[i]
    assert SB.sagebwd_workspace_bytes(1, 1, 100, 96) == 0
    assert SB.sagebwd_workspace_bytes(-1, 1, 100, 64) == 0
    assert SB.sagebwd_workspace_layout(1, 1, 100, 96)[0] == S.EINVAL


def test_fwd_and_bwd_reject_bad_arguments():
    B, H, N, D = 1, 2, 256, 64
    ws = 0x100000
    nb = SB.sagebwd_workspace_bytes(B, H, N, D)
    p = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000)
    fwd, bwd = SB.sagebwd_fwd, SB.sagebwd_bwd
    assert fwd(*p, B, H, N, 96, 0, 0.125, ws, nb, None) == S.EINVAL        # D
    assert fwd(*p, B, H, N, D, 2, 0.125, ws, nb, None) == S.EINVAL         # causal
    assert fwd(*p, B, H, N, D, 0, 0.0, ws, nb, None) == S.EINVAL           # scale
    assert fwd(*p, B, H, N, D, 0, float("nan"), ws, nb, None) == S.EINVAL
    assert fwd(*p, B, H, N, D, 0, 0.125, ws + 16, nb, None) == S.EINVAL    # workspace alignment
    assert fwd(*p, B, H, N, D, 0, 0.125, ws, nb - 1, None) == S.EINVAL     # workspace size
    assert fwd(0x1008, *p[1:], B, H, N, D, 0, 0.125, ws, nb, None) == S.EINVAL
    assert fwd(*p[:4], 0x5002, B, H, N, D, 0, 0.125, ws, nb, None) == S.EINVAL
    assert fwd(*p, B, H, 0, D, 0, 0.125, ws, SB.sagebwd_workspace_bytes(B, H, 0, D), None) == S.OK
    q = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000)
    assert bwd(*q, B, H, N, 96, 0, 0.125, ws, nb, None) == S.EINVAL
    assert bwd(*q, B, H, N, D, 0, -1.0, ws, nb, None) == S.EINVAL
    assert bwd(*q, B, H, N, D, 0, 0.125, ws, nb - 256, None) == S.EINVAL
    assert bwd(*q[:5], 0x6008, B, H, N, D, 0, 0.125, ws, nb, None) == S.EINVAL
    assert bwd(*q, 0, H, N, D, 1, 0.125, ws, SB.sagebwd_workspace_bytes(0, H, N, D), None) == S.OK
    # the step calls check the same way
    assert SB.sagebwd_quantize_qkv(0x1008, 0x2000, 0x3000, B, H, N, D, ws, nb, None) == S.EINVAL
    assert SB.sagebwd_quantize_qkv(*p[:3], B, H, N, 80, ws, nb, None) == S.EINVAL
    assert SB.sagebwd_attn_fwd(0x4000, 0x5002, B, H, N, D, 0, 0.125, ws, nb, None) == S.EINVAL
    assert SB.sagebwd_attn_fwd(0x4000, 0x5000, B, H, N, D, 3, 0.125, ws, nb, None) == S.EINVAL
    assert SB.sagebwd_bwd_prep(0x1000, 0x2000, 0x3000, B, H, N, D, ws, nb - 1, None) == S.EINVAL
    assert SB.sagebwd_attn_bwd(0x1000, 0x2008, B, H, N, D, 1, 0.125, ws, nb, None) == S.EINVAL
    assert SB.sagebwd_attn_bwd(0x1000, 0x2000, B, H, N, D, 1, float("inf"), ws, nb, None) == S.EINVAL
    assert SB.sagebwd_dq_out(0x1000, B, H, N, D, ws + 128, nb, None) == S.EINVAL
    assert SB.sagebwd_dq_out(0x1000, B, H, 0, D, ws, SB.sagebwd_workspace_bytes(B, H, 0, D), None) == S.OK


def test_probe_and_status_argument_checks():
    assert SB.sagebwd_mma_peak(7, 1, 1, 0x1000, None) == S.EINVAL
    assert SB.sagebwd_mma_peak(-1, 1, 1, 0x1000, None) == S.EINVAL
    assert SB.sagebwd_mma_peak(2, 1, (1 << 20) + 1, 0x1000, None) == S.EINVAL
    assert SB.sagebwd_mma_peak(0, 0, 1, 0x1000, None) == S.EINVAL
    assert SB.sagebwd_mma_peak(0, 1, 0, 0x1000, None) == S.EINVAL
    assert SB.sagebwd_get_status(0x1010, 1, 1, 128, 64, None) == S.EINVAL
    assert SB.sagebwd_get_status(0x1000, 1, 1, 128, 96, None) == S.EINVAL
    assert SB.sagebwd_int_mma_probe(0x1000, 0x2000, 24, 0x3000, None) == S.EINVAL
    assert SB.sagebwd_int_mma_probe(0x1000, 0x2000, 8192, 0x3000, None) == S.EINVAL
    assert SB.sagebwd_int_mma_probe(0x1001, 0x2000, 32, 0x3000, None) == S.EINVAL
    assert SB.sagebwd_umma_mn_probe(0x1001, 0x2000, 0x3000, 0x4000, None) == S.EINVAL
    assert SB.sagebwd_umma_ta_probe(0x1000, 0x2000, 96, 0x3000, 0x4000, None) == S.EINVAL
    assert SB.sagebwd_umma_ta_probe(0x1000, 0x2008, 64, 0x3000, 0x4000, None) == S.EINVAL
    assert SB.sagebwd_umma_mn_probe(0x1000, 0x2000, 0x3002, 0x4000, None) == S.EINVAL
    nb = SB.sagebwd_workspace_bytes(1, 2, 256, 64)
    st = SB.sagebwd_stall_test
    assert st(2, 0x1000, 0x2000, 1, 2, 256, 64, 0.125, 10 ** 7, 0x100000, nb, None) == S.EINVAL     # kernel
    assert st(0, 0x1000, 0x2000, 1, 2, 256, 64, 0.125, 10 ** 5, 0x100000, nb, None) == S.EINVAL     # limit < 1 ms
    assert st(0, 0x1000, 0x2000, 1, 2, 256, 64, 0.125, 2 * 10 ** 9, 0x100000, nb, None) == S.EINVAL
    assert st(0, 0x1000, 0x2002, 1, 2, 256, 64, 0.125, 10 ** 7, 0x100000, nb, None) == S.EINVAL     # lse alignment
    assert st(1, 0x1000, 0x2004, 1, 2, 256, 64, 0.125, 10 ** 7, 0x100000, nb, None) == S.EINVAL     # dv alignment
    assert st(0, 0x1000, 0x2000, 1, 2, 0, 64, 0.125, 10 ** 7, 0x100000, nb, None) == S.EINVAL       # empty
