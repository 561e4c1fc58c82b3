"""The whole path from host memory (sage_fp4_attention_host).

Q, K, V start in pinned host memory and O ends there; the library pipelines
chunks of heads through device staging slots on its own streams.  Every head
is computed by the same kernels as in the device-memory path, so O must be
bit-identical to sage_fp4_quantize_qkv + sage_fp4_attn_fwd on the same
inputs: checked for chunkings with a ragged last chunk, fewer heads than
chunks, ragged N, causal and D = 64, on a non-default stream, and for two
calls in a row that share one workspace.
"""
import pytest
import torch

from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300.synth import make_qkv

pytestmark = pytest.mark.gpu


def _device_path(q, k, v, causal):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    return S.attn_fwd(S.quantize_qkv(qd, kd, vd), causal).cpu()


@pytest.mark.parametrize("B,H,N,D,causal", [
    (2, 5, 300, 128, False),   # 10 heads: chunks of 2
    (3, 3, 700, 128, True),    # 9 heads: chunks of 2, last chunk of 1
    (1, 3, 1000, 64, True),    # fewer heads than chunks: one head per chunk
    (1, 1, 129, 64, False),    # a single head, N one past a tile
    (4, 32, 512, 128, True),   # 128 heads: 8 chunks of 16
])
def test_host_path_matches_device_path(B, H, N, D, causal):
    q, k, v = (t.pin_memory() for t in make_qkv(B, H, N, D, "k_channel_outliers", seed=B * N + D))
    want = _device_path(q, k, v, causal)
    ws = S.HostWorkspace(B, H, N, D)
    o = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16).pin_memory()
    S.attention_host(q, k, v, causal, out=o, workspace=ws)
    assert ws.get_status() == S.OK
    assert torch.equal(o, want)


def test_host_path_on_a_side_stream_two_calls_sharing_a_workspace():
    B, H, N, D = 2, 8, 640, 128
    ws = S.HostWorkspace(B, H, N, D)
    side = torch.cuda.Stream()
    ins = [tuple(t.pin_memory() for t in make_qkv(B, H, N, D, pat, seed=s))
           for s, pat in ((1, "k_channel_outliers"), (2, "iid"))]
    outs = [torch.empty((B, H, N, D), dtype=torch.bfloat16).pin_memory() for _ in ins]
    for (q, k, v), o in zip(ins, outs):  # queued back to back, no host sync between
        S.attention_host(q, k, v, False, out=o, workspace=ws, stream=side)
    side.synchronize()
    assert ws.get_status(side) == S.OK
    for (q, k, v), o in zip(ins, outs):
        assert torch.equal(o, _device_path(q, k, v, False))
