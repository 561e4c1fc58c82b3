"""Stream capture and determinism.

The calls are asynchronous on the caller's stream and allocate nothing, so a
whole quantize + attention step can be captured in a CUDA graph and replayed;
the host-memory pipeline forks its streams from the caller's stream and joins
them back, so it captures too.  The persistent schedule is static, so two
runs on the same inputs give the same bits.
"""
import pytest
import torch

from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300.synth import make_qkv

pytestmark = pytest.mark.gpu


def test_quantize_and_attention_replay_from_a_graph():
    B, H, N, D = 2, 4, 700, 128
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "k_channel_outliers", seed=41))
    z = S.QuantizedQKV(B, H, N, D)
    o = torch.empty_like(q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm up (first-call attribute setup) outside capture
        S.quantize_qkv(q, k, v, out=z, stream=side)
        S.attn_fwd(z, True, out=o, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = o.clone()
    g = torch.cuda.CUDAGraph()
    o.zero_()
    with torch.cuda.graph(g):
        S.quantize_qkv(q, k, v, out=z)
        S.attn_fwd(z, True, out=o)
    for _ in range(3):
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, want)
    assert z.get_status() == 0


def test_host_pipeline_replays_from_a_graph():
    B, H, N, D = 1, 8, 512, 64
    q, k, v = (t.pin_memory() for t in make_qkv(B, H, N, D, "iid", seed=42))
    ws = S.HostWorkspace(B, H, N, D)
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16).pin_memory()
    S.attention_host(q, k, v, False, out=o, workspace=ws)  # first call: streams, events
    torch.cuda.synchronize()
    want = o.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        S.attention_host(q, k, v, False, out=o, workspace=ws)
    for _ in range(2):
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, want)
    assert ws.get_status() == 0


def test_repeated_runs_are_bit_identical():
    B, H, N, D = 2, 8, 1000, 128
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "sparse_outliers", seed=43))
    runs = [S.attention(q, k, v, causal=c) for c in (False, False, True, True)]
    torch.cuda.synchronize()
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[2], runs[3])
