"""GPU parity of the NVFP4 decode matmul (aq_matmul_nvfp4_bf16) against the
oracle, through the C ABI."""
import numpy as np
import pytest

import affine_bit_quantized_gb300 as aq
import oracle
from affine_bit_quantized_gb300 import _build, synth

from ._helpers import assert_parity, from_dev_bf16, to_dev_bf16, to_dev_u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    _build.build_library()
    return torch.device("cuda:0")


def run(dev, x, w, pdl=False):
    import torch
    xt = to_dev_bf16(x, dev)
    wt = to_dev_u32(w.w_packed, dev)
    st = torch.from_numpy(np.ascontiguousarray(w.scales)).to(dev)
    y = aq.matmul_nvfp4(xt, wt, st, w.global_scale, pdl=pdl)
    torch.cuda.synchronize()
    return from_dev_bf16(y)


def check(dev, M, N, K, seed):
    w = synth.make_nvfp4_weights(N, K, seed)
    x = synth.make_x(M, K, seed)
    got = run(dev, x, w)
    _, ref = oracle.nvfp4_matmul(x, w.w_packed, w.scales, w.global_scale, M, N, K)
    assert aq.aq_read_device_status(None) == aq.AQ_OK
    return assert_parity(got, ref, what=f"nvfp4 M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 256), (1, 32, 256), (1, 33, 512), (1, 100, 2048), (1, 300, 2304), (1, 4096, 4096),
    (1, 64, 16384), (2, 77, 4096), (3, 129, 1280), (4, 50, 4096), (8, 64, 2048), (5, 31, 768),
    # x between 32 and 64 KB: the 3-stage ring beside it
    (8, 300, 4096), (2, 150, 14336), (1, 70, 32768), (7, 33, 4608), (3, 4096, 8192),
    # more rows than one CTA takes (8, or fewer for 64 KB of x): groups of CTAs that split the
    # rows and walk the same tiles, 8 row blocks per launch
    (16, 200, 4096), (12, 65, 2048), (5, 40, 14336), (9, 128, 32768),
    (16, 9760, 4096), (11, 3000, 14336), (20, 700, 32768), (70, 500, 4096),
])
def test_nvfp4_shapes(dev, M, N, K):
    check(dev, M, N, K, 900 + M + N + K)


def test_nvfp4_endpoints_and_nan(dev):
    """One-hot x returns global * scale * e2m1 of a column exactly (the weight
    is exact in fp16 and one product is exact in fp32); every code value and
    the extreme E4M3 scales appear; a NaN scale makes its outputs NaN."""
    N, K = 48, 512
    w = synth.make_nvfp4_weights(N, K, 21)
    w.w_packed[:8, 0] = 0x76543210                           # codes 0..7 at k = 0..7
    w.w_packed[8:16, 0] = 0xFEDCBA98                         # codes 8..15 (negative) at k = 0..7
    w.scales[:16, 0] = 0x7E                                    # 448
    w.scales[16, 0] = 0x01                                     # 2^-9, the smallest subnormal
    w.scales[17, 1] = 0x7F                                     # NaN
    for k in (0, 1, 3, 7):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        got = run(dev, x, w)
        _, ref = oracle.nvfp4_matmul(x, w.w_packed, w.scales, w.global_scale, 1, N, K)
        ok = ~np.isnan(oracle.bf16_to_double(ref[0]))
        assert np.array_equal(got[0][ok], ref[0][ok]), k
    x = synth.make_x(1, K, 22)
    got = run(dev, x, w)
    assert (got[0, 17] & 0x7F80) == 0x7F80 and (got[0, 17] & 0x7F)   # NaN


def test_nvfp4_pdl_and_deterministic(dev):
    M, N, K = 2, 1000, 4096
    w = synth.make_nvfp4_weights(N, K, 23)
    x = synth.make_x(M, K, 23)
    a = run(dev, x, w)
    b = run(dev, x, w, pdl=True)
    assert np.array_equal(a, b)


def test_nvfp4_lm_head_sampled(dev):
    """128256 x 4096 (the lm_head shape) at M = 1, sampled outputs."""
    N, K = synth.LLAMA8B_LM_HEAD[1], synth.LLAMA8B_LM_HEAD[2]
    w = synth.make_nvfp4_weights(N, K, 24)
    x = synth.make_x(1, K, 24)
    got = run(dev, x, w)
    rng = np.random.default_rng(24)
    inn = np.concatenate([rng.integers(0, N, 3000), [N - 1]])
    im = np.zeros_like(inn)
    ye, yb = oracle.nvfp4_matmul_sampled(x, w.w_packed, w.scales, w.global_scale, 1, N, K, im, inn)
    rms = float(np.sqrt(np.mean(ye * ye)))
    assert_parity(got[0, inn], yb, rms=rms, what="nvfp4 lm_head sampled")
