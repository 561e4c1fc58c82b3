"""Failure detection of the kernels' bounded waits, without a GPU fault.

sage_fp4_attn_fwd_stall_test runs the real kernel with its K-tile producer
stopping after the first KV tile of each CTA's stream, so the S issuer's
bounded wait for the next tile runs out.  The kernel must then abandon its
work through the normal drain path and report SAGE_FP4_ETIMEOUT in the status
word; the context must stay usable: a later launch that shares the set status
word skips its work, and after the status is read (and so reset) the same
operands give the same O as before.  sage_fp4_quantize_qkv_stall_test does
the same for the V quantizer's bounded wait for a copied tile.
"""
import time

import pytest
import torch

from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300.synth import make_qkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,D,causal", [(1, 2, 512, 128, False), (1, 1, 300, 64, True)])
def test_stalled_tile_sets_timeout_and_context_survives(B, H, N, D, causal):
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "iid", seed=3))
    z = S.quantize_qkv(q, k, v)
    ref = S.attn_fwd(z, causal)
    st = S._stream()
    assert z.get_status() == S.OK

    o = torch.zeros_like(q)
    t0 = time.time()
    rc = S.sage_fp4_attn_fwd_stall_test(z.struct, o.data_ptr(), B, H, N, D, causal, 20_000_000, st)
    assert rc == S.OK
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    # the wait gave up after its 20 ms limit, not the default 1.5 s
    assert elapsed < 1.0, elapsed

    # a launch that shares the set status word does no work
    o2 = torch.zeros_like(q)
    assert S.sage_fp4_attn_fwd(z.struct, o2.data_ptr(), B, H, N, D, int(causal), st) == S.OK
    torch.cuda.synchronize()
    assert int(o2.abs().sum().item()) == 0

    # reading the status resets it; the same operands then give the same O
    assert z.get_status() == S.ETIMEOUT
    assert z.get_status() == S.OK
    again = S.attn_fwd(z, causal)
    torch.cuda.synchronize()
    assert z.get_status() == S.OK
    assert torch.equal(again, ref)


def test_stall_test_rejects_limits_out_of_range():
    B, H, N, D = 1, 1, 128, 64
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "iid", seed=0))
    z = S.quantize_qkv(q, k, v)
    o = torch.empty_like(q)
    st = S._stream()
    for bad in (0, 999_999, 1_500_000_001):
        assert S.sage_fp4_attn_fwd_stall_test(z.struct, o.data_ptr(), B, H, N, D, 0, bad, st) == S.EINVAL
    assert z.get_status() == S.OK


@pytest.mark.parametrize("B,H,N,D", [(1, 2, 512, 128), (2, 3, 1000, 64), (1, 8, 8192, 128)])
def test_stalled_v_tile_sets_timeout_and_quantizer_recovers(B, H, N, D):
    # sage_fp4_quantize_qkv_stall_test: one block of the V quantizer never gets
    # its first tile, so its bounded wait runs out (20 ms); the whole block
    # leaves together, the status word reads ETIMEOUT, and the context stays
    # usable: after the status is read (and so reset), the same inputs give
    # the same quantized operands, byte for byte, as before the stall
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "iid", seed=4))
    z = S.quantize_qkv(q, k, v)
    torch.cuda.synchronize()
    assert z.get_status() == S.OK
    ref = z.workspace.clone()
    st = S._stream()
    t0 = time.time()
    rc = S.sage_fp4_quantize_qkv_stall_test(q.data_ptr(), k.data_ptr(), v.data_ptr(), z.struct, B, H, N, D,
                                            20_000_000, st)
    assert rc == S.OK
    torch.cuda.synchronize()
    assert time.time() - t0 < 1.0
    assert z.get_status() == S.ETIMEOUT
    assert z.get_status() == S.OK
    S.quantize_qkv(q, k, v, out=z)
    torch.cuda.synchronize()
    assert z.get_status() == S.OK
    assert torch.equal(z.workspace, ref)


def test_quantize_stall_test_rejects_limits_out_of_range():
    B, H, N, D = 1, 1, 128, 64
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "iid", seed=0))
    z = S.quantize_qkv(q, k, v)
    st = S._stream()
    for bad in (0, 999_999, 1_500_000_001):
        assert S.sage_fp4_quantize_qkv_stall_test(q.data_ptr(), k.data_ptr(), v.data_ptr(), z.struct, B, H, N,
                                                  D, bad, st) == S.EINVAL
    assert z.get_status() == S.OK
