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
    y = aq.matmul(xt, wt, st, bt, kernel=kernel, bits=w.bits)
    torch.cuda.synchronize()
    return from_dev_bf16(y)


def check_full(dev, M, N, K, seed, kernel="qmm", bits=4):
    w = synth.make_weights(N, K, seed, bits=bits)
    x = synth.make_x(M, K, seed)
    got = run(dev, x, w, kernel)
    _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, bits=bits)
    return assert_parity(got, ref, what=f"qmm M={M} N={N} K={K} bits={bits}")


def check_sampled(dev, M, N, K, seed, samples=3000, kernel="qmm", bits=4):
    w = synth.make_weights(N, K, seed, bits=bits)
    x = synth.make_x(M, K, seed)
    got = run(dev, x, w, kernel)
    rng = np.random.default_rng(seed)
    im = rng.integers(0, M, samples)
    inn = rng.integers(0, N, samples)
    # always include the tile corners and the last row/column
    im = np.concatenate([im, [0, M - 1, M - 1, 0, min(255, M - 1), min(256, M - 1)]])
    inn = np.concatenate([inn, [0, N - 1, 0, N - 1, min(255, N - 1), min(256, N - 1)]])
    ye, yb = oracle.matmul_sampled(x, w.w_packed, w.scales, w.biases, M, N, K, im, inn, bits=bits)
    rms = float(np.sqrt(np.mean(ye * ye)))
    return assert_parity(got[im, inn], yb, rms=rms, what=f"qmm sampled M={M} N={N} K={K} bits={bits}")


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


# ---------------------------------------------------------------- 8-bit codes (128-row x tiles)

@pytest.mark.parametrize("M,N,K", [
    (128, 256, 512), (17, 64, 512), (129, 300, 1024), (255, 513, 1536), (300, 700, 2048), (1, 100, 512),
    (1000, 257, 4096),
])
def test_qmm_eight_bit(dev, M, N, K):
    check_full(dev, M, N, K, 900 + M + N + K, bits=8)


@pytest.mark.parametrize("M", [256, 2048])
@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096)])
def test_qmm_eight_bit_prefill_shapes(dev, M, K, N):
    check_sampled(dev, M, N, K, 950 + M + K, bits=8)


def test_qmm_eight_bit_endpoints(dev):
    """8-bit codes on the tensor-core path: a one-hot x over a q = 0 column gives
    the bias and over a q = 255 column gives 255*scale + bias (each rounded to
    fp16 on chip, then to bf16: compared with the oracle under the usual bound);
    auto selects this path above 16 rows."""
    N, K, M = 300, 1024, 40
    w = synth.make_weights(N, K, 23, bits=8)
    codes = oracle.unpack(w.w_packed, N, K, 8)
    codes[:, 3] = 0
    codes[:, 900] = 255
    w.w_packed = oracle.pack(codes, 8)
    x = synth.make_x(M, K, 23)
    x[0] = 0
    x[0, 3] = 0x3F80
    x[1] = 0
    x[1, 900] = 0x3F80
    got = run(dev, x, w, kernel="auto")
    _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, bits=8)
    assert_parity(got, ref, what="8-bit endpoints")
    assert np.array_equal(got[0], w.biases[:, 0])


@pytest.mark.parametrize("M,N,K,bits", [(256, 512, 4096, 4), (64, 256, 8192, 4), (128, 300, 4096, 8)])
def test_qmm_split_k(dev, M, N, K, bits):
    """Few output tiles: K is split across a cluster of CTAs whose partial tiles
    are added in shared memory in a fixed order.  Against the oracle, and the
    same bits on every call."""
    import torch
    check_full(dev, M, N, K, 1300 + M + K, bits=bits)
    w = synth.make_weights(N, K, 7, bits=bits)
    x = synth.make_x(M, K, 7)
    xt, wt, st, bt = upload(x, w, dev)
    y1 = aq.matmul(xt, wt, st, bt, kernel="qmm", bits=bits)
    y2 = aq.matmul(xt, wt, st, bt, kernel="qmm", bits=bits)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("M,N,K,bits", [
    (512, 256, 512, 4), (1100, 300, 512, 4), (2048, 600, 512, 4),    # 256-row tiles; 5 row tiles: one padding CTA
    (512, 300, 512, 8), (640, 257, 512, 8), (1300, 520, 512, 8),     # 128-row tiles
    (512, 4864, 512, 4), (640, 2600, 512, 8),                        # W the larger operand: row tiles fastest
])
def test_qmm_cta_pairs(dev, M, N, K, bits):
    """Without a K split (K = 512: one block of 8 groups) and with at least two
    row tiles of x, CTA pairs share each W tile: each converts half of it and
    one MMA over 256 rows of x spans both.  Every output against the oracle,
    with ragged M and N and a pair whose second CTA has no rows of x."""
    check_full(dev, M, N, K, 1500 + M + N, bits=bits)


@pytest.mark.parametrize("M,N,K,bits", [(256, 256, 512, 4), (256, 512, 4096, 4), (512, 256, 512, 4),
                                        (512, 300, 512, 8)])   # one CTA; split K; CTA pairs
def test_qmm_pdl_flag_same_bits(dev, M, N, K, bits):
    """Programmatic dependent launch beside the cluster launch of a K split or a
    CTA pair: the same bits as a plain launch, after a preceding kernel that
    writes x on the same stream."""
    import torch
    w = synth.make_weights(N, K, 1600 + M, bits=bits)
    x = synth.make_x(M, K, 1600 + M)
    xt, wt, st, bt = upload(x, w, dev)
    a = aq.matmul(xt, wt, st, bt, kernel="qmm", bits=bits)
    x2 = torch.zeros_like(xt)
    x2.copy_(xt)                     # the kernel before the launch writes its x
    b = aq.matmul(x2, wt, st, bt, kernel="qmm", bits=bits, pdl=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert aq.aq_read_device_status(torch.cuda.current_stream().cuda_stream) == aq.AQ_OK


@pytest.mark.parametrize("M,N,K,bits", [
    (17, 64, 512, 4), (300, 700, 2048, 4), (256, 512, 4096, 4), (2048, 1024, 4096, 4),
    (129, 300, 1024, 8), (1000, 257, 4096, 8),
    (1024, 300, 512, 4), (640, 257, 512, 8), (2048, 4864, 512, 8),   # CTA pairs without the workspace
    (2048, 4096, 512, 8), (2048, 4096, 14336, 8),   # with it: 224-row tiles, stages laid out for 224 rows
])
def test_qmm_workspace_path_same_bits(dev, M, N, K, bits):
    """With a workspace, x is converted to fp16 once and copied straight into
    the MMA tiles: the same bits as without (also where the call without the
    workspace runs on CTA pairs and the one with it on single CTAs), and the
    oracle's result class."""
    import torch
    w = synth.make_weights(N, K, 1400 + M, bits=bits)
    x = synth.make_x(M, K, 1400 + M)
    xt, wt, st, bt = upload(x, w, dev)
    ws = torch.empty(aq.aq_matmul_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
    assert ws.numel() == M * K * 2
    a = aq.matmul(xt, wt, st, bt, bits=bits)
    b = aq.matmul(xt, wt, st, bt, bits=bits, workspace=ws)
    b2 = aq.matmul(xt, wt, st, bt, bits=bits, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(b, b2), "the workspace path is not deterministic"
    diff = (a.view(torch.int16) != b.view(torch.int16))
    assert not diff.any(), f"{int(diff.sum())} of {diff.numel()} outputs differ, rows {diff.any(1).nonzero()[:8].flatten().tolist()}"
    if M * N <= 300 * 700:
        _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, bits=bits)
        assert_parity(from_dev_bf16(b), ref, what=f"qmm workspace M={M} N={N} K={K}")


def test_output_beyond_2_31_elements(dev):
    """A prefill over a vocabulary-sized N: y has 2.7e9 elements (5.4 GB), so
    the outputs past row 2^31 / N sit at offsets that need 64 bits.  Sampled
    outputs, half of them past that row, are gathered on the device."""
    import torch
    M, N, K = 20480, 131072, 512
    w = synth.make_weights(N, K, 77)
    x = synth.make_x(M, K, 77)
    xt, wt, st, bt = upload(x, w, dev)
    y = aq.matmul(xt, wt, st, bt)
    hi = (1 << 31) // N                      # first row whose offset reaches 2^31
    rng = np.random.default_rng(77)
    im = np.concatenate([rng.integers(0, hi, 1000), rng.integers(hi, M, 2000), [hi, hi, M - 1, M - 1]])
    inn = np.concatenate([rng.integers(0, N, 3000), [0, N - 1, 0, N - 1]])
    got = from_dev_bf16(y[torch.from_numpy(im).to(dev), torch.from_numpy(inn).to(dev)])
    torch.cuda.synchronize()
    del y
    ye, yb = oracle.matmul_sampled(x, w.w_packed, w.scales, w.biases, M, N, K, im, inn)
    rms = float(np.sqrt(np.mean(ye * ye)))
    assert_parity(got, yb, rms=rms, what=f"qmm sampled M={M} N={N} K={K} (y beyond 2^31 elements)")


@pytest.mark.parametrize("M,N,K,bits", [(64, 512, 1024, 4), (256, 512, 4096, 4),   # one tile; split K over a cluster
                                        (512, 256, 512, 4),                        # a CTA pair
                                        (512, 256, 512, 8),                        # a pair converting x in its stages
                                        (256, 512, 4096, 8)])                      # 8-bit, split K, three raw stages
def test_qmm_bounded_wait_timeout_reports_status(dev, M, N, K, bits):
    """The test hook makes the first CTA's producer leave out its first copy:
    the converters' bounded wait expires, the kernel records a timeout (the
    other CTAs of a split-K cluster still meet it at the cluster barriers; the
    other CTA of a pair waits out its own bounded waits for the stages that
    never get consumed), the host reads AQ_ERR_TIMEOUT, and a normal call
    right after is correct."""
    import torch
    w = synth.make_weights(N, K, 12, bits=bits)
    x = synth.make_x(M, K, 12)
    xt, wt, st, bt = upload(x, w, dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert aq.aq_read_device_status(stream) == aq.AQ_OK
    aq.matmul(xt, wt, st, bt, kernel="qmm", bits=bits, flags=aq.AQ_FLAG_DEBUG_SKIP_COPY)
    assert aq.aq_read_device_status(stream) == aq.AQ_ERR_TIMEOUT
    assert aq.aq_read_device_status(stream) == aq.AQ_OK          # cleared by the read
    check_full(dev, M, N, K, 12, bits=bits)
