"""Device primitives pinned against the oracle and exact arithmetic.

* Every float32 bit pattern through the device E2M1 / E4M3 conversions the
  kernels use, compared with the oracle's codecs (NaN inputs are outside the
  contract and only reported).
* One block-scaled FP4 tensor-core product of a 128-row tile against an
  exact float64 product of the decoded operands: E2M1 x E2M1 x E4M3 x E4M3
  products are exact in FP32, so only the FP32 accumulation order differs.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_attention_gb300 import sage_fp4 as S
from helpers import e2m1_table, plain_to_block

pytestmark = pytest.mark.gpu


def test_cvt_probe_all_float32_patterns():
    chunk = 1 << 28
    e2 = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    e4 = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    nan_e4 = set()
    for first in range(0, 1 << 32, chunk):
        rc = S.sage_fp4_cvt_probe(first, chunk, e2.data_ptr(), e4.data_ptr(), stream)
        assert rc == 0
        g2 = e2.cpu().numpy()
        g4 = e4.cpu().numpy()
        r2, r4 = oracle.encode_range(first, chunk)
        bits = np.arange(first, first + chunk, dtype=np.uint64).astype(np.uint32)
        nan = ((bits >> 23) & 0xFF) == 0xFF
        nan &= (bits & 0x7FFFFF) != 0
        ok2 = (g2 == r2) | nan
        ok4 = (g4 == r4) | nan
        if not ok2.all():
            i = int(np.flatnonzero(~ok2)[0])
            raise AssertionError(f"E2M1 mismatch at bits {int(bits[i]):#010x}: gpu {g2[i]:#x} oracle {r2[i]:#x}")
        if not ok4.all():
            i = int(np.flatnonzero(~ok4)[0])
            raise AssertionError(f"E4M3 mismatch at bits {int(bits[i]):#010x}: gpu {g4[i]:#x} oracle {r4[i]:#x}")
        if nan.any():
            nan_e4 |= set(np.unique(g4[nan]).tolist())
    print("E4M3 of NaN inputs:", sorted(nan_e4))


def _rand_operand(rng, rows, K, rows_pad=128):
    codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
    # scales between 2^-4 and 2^4 keep every product well inside FP32
    sc = rng.integers(0x20, 0x58, size=(rows, K // 16), dtype=np.uint8)
    plain = np.zeros((rows_pad, K // 16), np.uint8)
    plain[:rows] = sc
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    e4 = np.array([oracle.e4m3_value(b) for b in range(256)])
    dec = e2m1_table()[codes] * np.repeat(e4[sc], 16, axis=1)
    return packed, plain_to_block(plain), dec


@pytest.mark.parametrize("K", [64, 128, 256])
@pytest.mark.parametrize("n", [64, 128])
@pytest.mark.parametrize("a_by_threads", [0, 1])
@pytest.mark.parametrize("sf_rows128", [0, 1])
def test_mma_probe_exact_product(K, n, a_by_threads, sf_rows128):
    # sf_rows128: A row r's scales in lane r alone (column base + r / 32), noise elsewhere
    rng = np.random.default_rng(K * 7 + n + a_by_threads)
    a_codes, a_sf, a_dec = _rand_operand(rng, 128, K)
    b_codes, b_sf, b_dec = _rand_operand(rng, n, K)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    ta, tsa, tb, tsb = dev(a_codes), dev(a_sf), dev(b_codes), dev(b_sf)
    d = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = (S.PROBE_A_BY_THREADS if a_by_threads else 0) | (S.PROBE_SF_ROWS128 if sf_rows128 else 0)
    rc = S.sage_fp4_mma_probe_ex(ta.data_ptr(), tsa.data_ptr(), tb.data_ptr(), tsb.data_ptr(), n, K,
                                 flags, d.data_ptr(), status.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = d.cpu().numpy().astype(np.float64)
    ref = a_dec @ b_dec.T
    scale = np.abs(a_dec) @ np.abs(b_dec).T
    err = np.abs(got - ref) / np.maximum(scale, 1e-30)
    assert np.isfinite(got).all()
    assert err.max() < 1e-5, (err.max(), np.unravel_index(err.argmax(), err.shape))


@pytest.mark.parametrize("n", [128, 256])
def test_mma_peak_rate(n):
    # back-to-back FP4 MMAs on every SM: a plausible dense FP4 rate for one
    # GB300 (the nominal dense NVFP4 figure is 13.5-15 PFLOP/s at full clock)
    tflops = S.mma_peak_tflops(n=n, iters=4000)
    print(f"FP4 MMA rate, N={n}: {tflops:.0f} TFLOP/s")
    assert 3000 < tflops < 20000, tflops


def test_tmem_reducing_load_gives_group_maxima():
    # The attention kernel takes each 16-key group's maximum of a score row
    # from the load that brings the scores out of tensor memory.  Pin what it
    # returns: the values unchanged, and per 16 columns their maximum --
    # including -inf (masked keys), groups of equal values, +-0 and values of
    # every magnitude a score can take.
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((128, 128)) * np.exp(rng.uniform(-20, 20, (128, 1)))).astype(np.float32)
    x[1, :16] = -np.inf                # a fully masked group
    x[2, 5:16] = -np.inf               # a partly masked group
    x[3, 16:32] = 2.5                  # equal values
    x[4, 32:48] = -0.0
    x[5, 48:64] = -rng.uniform(1, 2, 16).astype(np.float32)  # all negative
    x[6, 64] = 3.0e38
    xin = torch.from_numpy(x).cuda()
    vals = torch.full((128, 128), float("nan"), device="cuda")
    maxes = torch.full((128, 8), float("nan"), device="cuda")
    rc = S.sage_fp4_tmem_max_probe(xin.data_ptr(), vals.data_ptr(), maxes.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == S.OK, S.strerror(rc)
    torch.cuda.synchronize()
    v, m = vals.cpu().numpy(), maxes.cpu().numpy()
    assert np.array_equal(v.view(np.uint32), x.view(np.uint32))
    want = x.reshape(128, 8, 16).max(-1)
    assert np.array_equal(m, want), np.argwhere(m != want)[:5]
