"""The pages' one format comparison, on the synthetic stand-ins.

[NEWS-HW] compares MXFP4 and NVFP4 on real Q, K, V from every layer of
CogVideoX and keeps NVFP4, which is much more accurate.  Those activations are
not available; here each benchmark workload's value pattern (at its own N and
D, two heads, 96 sampled query rows) is attended by the oracle's method in
both formats and compared with exact float64 attention.  NVFP4 must come out
ahead on every pattern, in cosine similarity and in relative L1.

Measured (seed 0; cosine / relative L1, NVFP4 then MXFP4):
  iid N512 D128                      0.983 / 0.185   0.971 / 0.232
  K channel outliers N4096 D128      0.857 / 0.616   0.584 / 1.005
  same, causal N8192                 0.715 / 0.759   0.668 / 0.940
  K head mean N17776 D64             0.947 / 0.320   0.932 / 0.354
  sparse outliers N32768 D128        0.928 / 0.316   0.723 / 0.646
"""
import numpy as np
import pytest

import oracle
from bit_attention_gb300.synth import WORKLOADS, make_qkv


def _errors(o, ex):
    cos = float((o * ex).sum() / np.sqrt((o * o).sum() * (ex * ex).sum()))
    return cos, float(np.abs(o - ex).sum() / np.abs(ex).sum())


@pytest.mark.parametrize("name", ["small", "llm", "llm_causal", "dit", "dit_long"])
def test_nvfp4_is_more_accurate_than_mxfp4(name):
    w = WORKLOADS[name]
    B, H = 1, 2
    q, k, v = make_qkv(B, H, w.N, w.D, w.pattern, seed=0)
    rows = np.sort(np.random.default_rng(0).choice(B * H * w.N, size=96, replace=False))
    exact = oracle.attention_exact(q, k, v, B * H, w.N, w.D, w.causal, rows=rows)
    res = {}
    for fmt in ("nvfp4", "mxfp4"):
        qz = oracle.Quantized(q, k, v, B * H, w.N, w.D, fmt=fmt)
        res[fmt] = _errors(oracle.attention(qz, w.causal, rows=rows)[0], exact)
    print(f"{name}: NVFP4 cos {res['nvfp4'][0]:.4f} L1 {res['nvfp4'][1]:.4f} | "
          f"MXFP4 cos {res['mxfp4'][0]:.4f} L1 {res['mxfp4'][1]:.4f}")
    assert res["nvfp4"][0] > res["mxfp4"][0] and res["nvfp4"][1] < res["mxfp4"][1], res
