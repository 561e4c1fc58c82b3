"""The one-call entry point that allocates nothing (sage_fp4_attention_noalloc).

It serves callers that cannot call cudaMalloc, such as code inside another
framework's operator without access to its allocator: they pass only q, k,
v, o and a status word, and the quantized operands live in the library's
fixed 64 MiB device array.  This file checks, through the C ABI, that two
calls in a row (different shapes, so the second reads over what the first
left in the shared array) give exactly the O of the two-call API
(sage_fp4_quantize_qkv + sage_fp4_attn_fwd with a workspace): the same
kernels run on the same operands, so the bits must agree.  It also checks
that an oversized problem is rejected.  This file is collected last, so that
a run stopping at the first failure has already run every other test.
"""
import pytest
import torch

from bit_attention_gb300 import sage_fp4 as S
from bit_attention_gb300.synth import make_qkv

pytestmark = pytest.mark.gpu


def test_noalloc_matches_two_call_api_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for B, H, N, D, causal, pattern in [(1, 4, 1000, 128, True, "k_channel_outliers"),
                                        (2, 3, 300, 64, False, "k_head_mean")]:
        q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, pattern, seed=N))
        ref = S.attn_fwd(S.quantize_qkv(q, k, v), causal)
        o = torch.full_like(q, float("nan"))
        rc = S.sage_fp4_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                          status.data_ptr(), B, H, N, D, causal, stream)
        assert rc == S.OK, S.strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(o, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # B4 H32 N4096 D128 needs 108 MiB of quantized operands: more than 64 MiB
    assert S.sage_fp4_workspace_bytes(4, 32, 4096, 128) > (64 << 20)
    rc = S.sage_fp4_attention_noalloc(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 4, 32, 4096, 128, 0,
                                      None)
    assert rc == S.ETOOLARGE
    assert "64 MiB" in S.strerror(rc)
