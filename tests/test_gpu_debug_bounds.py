"""The bounds-checking debug build (SAGE_FP4_DEBUG_BOUNDS=1, libsagefp4_debug.so).

Its kernels check every global-memory index they compute (the quantizers'
loads of Q, K, V and stores of codes and scales; the attention kernel's scale
copies and O stores) against the buffer it falls in; a failure is recorded as
SAGE_FP4_EBOUNDS in the status word and the access skipped, with no trap and
no device assert.  Over the layouts, formats and ragged shapes below it must
report nothing and produce exactly the release build's bytes.
"""
import pytest
import torch

from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300.synth import make_qkv

pytestmark = pytest.mark.gpu


def _path(q, k, v, causal, fmt, layout):
    if layout == "NHD":
        return None, S.attention(q, k, v, causal, layout="NHD", fmt=fmt)
    z = S.quantize_qkv(q, k, v, fmt=fmt)
    o = S.attn_fwd(z, causal)
    torch.cuda.synchronize()
    assert z.get_status() == S.OK
    return z, o


@pytest.mark.parametrize("B,H,N,D,causal,fmt,layout", [
    (1, 2, 300, 128, True, "nvfp4", "HND"),
    (2, 3, 777, 64, False, "nvfp4", "HND"),
    (1, 1, 17, 128, False, "mxfp4", "HND"),
    (2, 2, 1000, 64, True, "mxfp4_directp", "HND"),
    (2, 3, 333, 128, False, "nvfp4", "NHD"),
    (4, 32, 1024, 128, False, "nvfp4", "HND"),
])
def test_debug_build_reports_nothing_and_matches_release(B, H, N, D, causal, fmt, layout):
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "k_channel_outliers", seed=N + D))
    if layout == "NHD":
        q, k, v = (x.transpose(1, 2).contiguous() for x in (q, k, v))
    z, o = _path(q, k, v, causal, fmt, layout)
    with S.debug_bounds_library():
        zd, od = _path(q, k, v, causal, fmt, layout)
        torch.cuda.synchronize()
        if zd is not None:
            assert zd.get_status() == S.OK
    assert torch.equal(od, o)
    if z is not None:
        assert torch.equal(zd.workspace[:-256], z.workspace[:-256])
