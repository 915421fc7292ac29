"""GPU parity of the tensor-core path (tcgen05 qmm, M > 16 by default) against
the oracle, through the C ABI."""
import numpy as np
import pytest

import affine_bit_quantized_gb300 as aq
import oracle
from affine_bit_quantized_gb300 import _build, synth

from ._helpers import assert_parity, from_dev_bf16, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    _build.build_library()
    return torch.device("cuda:0")


def run(dev, x, w, kernel="qmm"):
    import torch
    xt, wt, st, bt = upload(x, w, dev)
    y = aq.matmul(xt, wt, st, bt, kernel=kernel)
    torch.cuda.synchronize()
    return from_dev_bf16(y)


def check_full(dev, M, N, K, seed, kernel="qmm"):
    w = synth.make_weights(N, K, seed)
    x = synth.make_x(M, K, seed)
    got = run(dev, x, w, kernel)
    _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K)
    return assert_parity(got, ref, what=f"qmm M={M} N={N} K={K}")


def check_sampled(dev, M, N, K, seed, samples=3000, kernel="qmm"):
    w = synth.make_weights(N, K, seed)
    x = synth.make_x(M, K, seed)
    got = run(dev, x, w, kernel)
    rng = np.random.default_rng(seed)
    im = rng.integers(0, M, samples)
    inn = rng.integers(0, N, samples)
    # always include the tile corners and the last row/column
    im = np.concatenate([im, [0, M - 1, M - 1, 0, min(255, M - 1), min(256, M - 1)]])
    inn = np.concatenate([inn, [0, N - 1, 0, N - 1, min(255, N - 1), min(256, N - 1)]])
    ye, yb = oracle.matmul_sampled(x, w.w_packed, w.scales, w.biases, M, N, K, im, inn)
    rms = float(np.sqrt(np.mean(ye * ye)))
    return assert_parity(got[im, inn], yb, rms=rms, what=f"qmm sampled M={M} N={N} K={K}")


def test_qmm_single_tile(dev):
    check_full(dev, 256, 256, 512, 31)


@pytest.mark.parametrize("M,N,K", [
    (17, 64, 512), (64, 300, 1024), (100, 256, 512), (255, 513, 1536), (257, 256, 512), (300, 700, 2048),
    (1, 100, 512), (5, 33, 1024), (512, 1000, 4096),
])
def test_qmm_ragged(dev, M, N, K):
    check_full(dev, M, N, K, M + N + K)


@pytest.mark.parametrize("M", [256, 2048])
@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096)])
def test_prefill_config(dev, M, K, N):
    check_sampled(dev, M, N, K, synth.seed_for(5, M // 256, 0 if N == 14336 else 1))


def test_auto_selects_tensor_core_path_above_16_rows(dev):
    # M = 17 by default runs the tensor-core kernel; same result class as the oracle
    check_full(dev, 17, 129, 1024, 5, kernel="auto")


def test_qmm_deterministic(dev):
    import torch
    M, N, K = 300, 512, 2048
    w = synth.make_weights(N, K, 3)
    x = synth.make_x(M, K, 3)
    xt, wt, st, bt = upload(x, w, dev)
    a = aq.matmul(xt, wt, st, bt, kernel="qmm")
    b = aq.matmul(xt, wt, st, bt, kernel="qmm")
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert aq.aq_read_device_status(None) == aq.AQ_OK
