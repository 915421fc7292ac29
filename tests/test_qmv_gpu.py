"""GPU parity of the weight-streaming path (M = 1..16 and chunked larger M)
against the oracle, element by element, through the C ABI."""
import numpy as np
import pytest

import affine_bit_quantized_gb300 as aq
import oracle
from affine_bit_quantized_gb300 import _build, synth

from ._helpers import assert_parity, bf16_to_f64, from_dev_bf16, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    _build.build_library()
    return torch.device("cuda:0")


def run(dev, x, w, kernel="qmv", pdl=False):
    import torch
    xt, wt, st, bt = upload(x, w, dev)
    y = aq.matmul(xt, wt, st, bt, kernel=kernel, pdl=pdl, bits=w.bits)
    torch.cuda.synchronize()
    return from_dev_bf16(y)


def check(dev, M, N, K, seed, kernel="qmv", pdl=False, bits=4):
    w = synth.make_weights(N, K, seed, bits=bits)
    x = synth.make_x(M, K, seed)
    got = run(dev, x, w, kernel, pdl)
    _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, bits=bits)
    return assert_parity(got, ref, what=f"M={M} N={N} K={K} bits={bits}")


def test_tiny_correctness_config(dev):
    # 256 x 512 weights, M = 1, seed 0
    check(dev, 1, 256, 512, synth.seed_for(1))


@pytest.mark.parametrize("name,N,K", synth.LLAMA8B_LAYER + (synth.LLAMA8B_LM_HEAD,))
def test_llama8b_layer_m1(dev, name, N, K):
    j = [n for n, _, _ in synth.LLAMA8B_LAYER + (synth.LLAMA8B_LM_HEAD,)].index(name)
    check(dev, 1, N, K, synth.seed_for(2, 0, j))


@pytest.mark.parametrize("M", [2, 4, 8, 16])
@pytest.mark.parametrize("name,N,K", [s for s in synth.LLAMA8B_LAYER if s[0] in ("q_proj", "k_proj", "down_proj")])
def test_small_batch_sweep(dev, M, name, N, K):
    j = [n for n, _, _ in synth.LLAMA8B_LAYER].index(name)
    check(dev, M, N, K, synth.seed_for(3, M, j))


@pytest.mark.parametrize("M,kernel", [(2, "qmv"), (16, "qmv"), (16, "auto"), (12, "auto"), (9, "auto")])
def test_small_batch_lm_head_sampled(dev, M, kernel):
    """The lm_head shape at small batch.  With "qmv", 9..16 rows run in one
    launch on the two blocks of MMA columns (in K passes: x of 16 rows of
    K = 4096 is 128 KB); with "auto", in one launch whose CTA pairs take the
    two halves of the rows."""
    import torch
    _, N, K = synth.LLAMA8B_LM_HEAD
    w = synth.make_weights(N, K, synth.seed_for(3, M, 7))
    x = synth.make_x(M, K, synth.seed_for(3, M, 7))
    got = run(dev, x, w, kernel=kernel)
    rng = np.random.default_rng(M)
    im = rng.integers(0, M, 4000)
    inn = rng.integers(0, N, 4000)
    ye, yb = oracle.matmul_sampled(x, w.w_packed, w.scales, w.biases, M, N, K, im, inn)
    rms = float(np.sqrt(np.mean(ye * ye)))
    assert_parity(got[im, inn], yb, rms=rms, what="lm_head sampled")


@pytest.mark.parametrize("M", [9, 10, 11, 12, 13, 14, 15, 16])
@pytest.mark.parametrize("N,K", [(100, 512), (300, 2048), (67, 4096), (40, 8704)])
def test_nine_to_sixteen_rows_one_pass(dev, M, N, K):
    """9..16 rows of x on the weight-streaming kernel's two blocks of MMA
    columns: ragged N, x in one pass (K <= 2048) and in K passes (K = 4096,
    8704 with a ragged last stage), element by element against the oracle, on
    the default choice and on the explicit one."""
    check(dev, M, N, K, 900 + M + K, kernel="auto")
    check(dev, M, N, K, 950 + M + K, kernel="qmv")


@pytest.mark.parametrize("M,N,K,bits", [
    (9, 9729, 4096, 4),     # halves of 5 and 4 rows; a ragged last tile
    (13, 10000, 4096, 4),
    (16, 9760, 4096, 4),    # 305 tiles over 76 pairs
    (16, 10016, 8192, 4),   # each half's x in two K passes
    (11, 9728, 4096, 8),
    (16, 9760, 2048, 8),
    (16, 4900, 4096, 4),    # 154 tiles: one per SM is enough where each half fits one pass
    (12, 2048, 4096, 8),    # 8-bit codes: over any number of tiles
    (16, 4096, 14336, 8),   # each half's x in K passes
    (12, 1024, 8192, 8),
    (9, 100, 4096, 8),      # 4 tiles: 4 CTA pairs
])
def test_nine_to_sixteen_rows_split_pairs(dev, M, N, K, bits):
    """9..16 rows over enough tiles, where x of all the rows would need K
    passes: the default choice is one launch whose CTA pairs take the two
    halves of x's rows and walk the same tiles; every output against the
    oracle."""
    check(dev, M, N, K, 990 + M + N + bits, kernel="auto", bits=bits)


def test_split_pairs_bounded_wait_timeout(dev):
    """The test hook on the split-rows launch: every CTA of both halves runs its
    bounded wait out, the host reads AQ_ERR_TIMEOUT, and a normal call right
    after is correct."""
    import torch
    M, N, K = 12, 9728, 4096
    w = synth.make_weights(N, K, 14)
    x = synth.make_x(M, K, 14)
    xt, wt, st, bt = upload(x, w, dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert aq.aq_read_device_status(stream) == aq.AQ_OK
    aq.matmul(xt, wt, st, bt, flags=aq.AQ_FLAG_DEBUG_SKIP_COPY)
    assert aq.aq_read_device_status(stream) == aq.AQ_ERR_TIMEOUT
    assert aq.aq_read_device_status(stream) == aq.AQ_OK
    check(dev, M, N, K, 14, kernel="auto")


@pytest.mark.parametrize("M,N,K", [(9, 70, 1024), (16, 300, 4096), (12, 33, 5120)])
def test_nine_to_sixteen_rows_eight_bit(dev, M, N, K):
    check(dev, M, N, K, 970 + M, bits=8)


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 64), (1, 14, 64), (1, 15, 64), (1, 16, 64), (1, 31, 128), (3, 45, 576), (5, 7, 1088),
    (8, 33, 4160), (9, 100, 192), (13, 256, 1024), (16, 15, 64), (1, 1000, 8192), (2, 77, 16384),
    (17, 50, 256), (33, 40, 512), (70, 31, 320),
])
def test_ragged_shapes(dev, M, N, K):
    check(dev, M, N, K, 100 + M + N + K)


@pytest.mark.parametrize("M,N,K,bits", [
    (2, 300, 16384, 4),    # x of 64 KB: two passes of 8192 codes
    (8, 77, 4096, 4),      # one 2048-code stage per pass
    (3, 1000, 14336, 4),   # four passes, the last of one stage
    (1, 100, 28672, 4),    # one row beyond 16384 codes: 8 stages, then 6
    (5, 4100, 6144, 4),    # three passes over 129 tiles
    (7, 33, 2560, 4),      # second pass of 512 codes (a partial stage)
    (4, 64, 33280, 4),     # nine passes, the last of 512 codes
    (8, 200, 4096, 8),
    (1, 64, 32768, 8),
    (3, 50, 7680, 8),      # second pass of 2560 codes
])
@pytest.mark.parametrize("kernel", ["qmv", "auto"])
def test_tma_kernel_k_passes(dev, M, N, K, bits, kernel):
    """x larger than one staging (M*K*2 > 32 KB): the TMA-fed kernel walks K
    in passes and keeps each tile's sums in shared memory across them ("qmv"
    forces it; "auto" may pick the general kernel for these shapes)."""
    check(dev, M, N, K, 600 + M + N + K, kernel=kernel, bits=bits)


def test_tma_kernel_tile_batches_sampled(dev):
    """8 rows of x over the 128256 x 4096 lm_head matrix with 8-bit codes: two
    K passes, and more tiles per CTA than the shared-memory tile sums hold, so
    the tiles go in batches.  Sampled outputs against the oracle."""
    _, N, K = synth.LLAMA8B_LM_HEAD
    M = 8
    w = synth.make_weights(N, K, 777, bits=8)
    x = synth.make_x(M, K, 777)
    got = run(dev, x, w)
    rng = np.random.default_rng(7)
    im = rng.integers(0, M, 4000)
    inn = np.concatenate([rng.integers(0, N, 3990), np.arange(N - 10, N)])
    ye, yb = oracle.matmul_sampled(x, w.w_packed, w.scales, w.biases, M, N, K, im, inn, bits=8)
    rms = float(np.sqrt(np.mean(ye * ye)))
    assert_parity(got[im, inn], yb, rms=rms, what="lm_head 8-bit M=8 sampled")


def test_pdl_flag_same_bits(dev):
    M, N, K = 4, 300, 1024
    w = synth.make_weights(N, K, 5)
    x = synth.make_x(M, K, 5)
    a = run(dev, x, w, pdl=False)
    b = run(dev, x, w, pdl=True)
    assert np.array_equal(a, b)


def test_deterministic(dev):
    import torch
    M, N, K = 3, 4096, 4096
    w = synth.make_weights(N, K, 6)
    x = synth.make_x(M, K, 6)
    xt, wt, st, bt = upload(x, w, dev)
    y1 = aq.matmul(xt, wt, st, bt)
    y2 = aq.matmul(xt, wt, st, bt)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_k_zero_writes_zeros_and_m_zero_is_noop(dev):
    import torch
    y = torch.full((2, 5), 3.0, dtype=torch.bfloat16, device=dev)
    p = y.data_ptr()
    st = aq.aq_matmul_bf16(p, p, p, p, p, 2, 5, 0, 64, 4, None)
    torch.cuda.synchronize()
    assert st == aq.AQ_OK and not y.float().any()
    y.fill_(3.0)
    st = aq.aq_matmul_bf16(p, p, p, p, p, 0, 5, 64, 64, 4, None)
    torch.cuda.synchronize()
    assert st == aq.AQ_OK and bool((y.float() == 3.0).all())


@pytest.mark.parametrize("K", [256, 1024])   # generic kernel, TMA-fed kernel
def test_special_inputs(dev, K):
    """Zero x gives exact zeros; a one-hot x returns one dequantized column
    (q = 0 gives the bias); NaN in x propagates to every output of its row."""
    N = 40
    w = synth.make_weights(N, K, 9)
    codes = oracle.unpack(w.w_packed, N, K)
    codes[:, 5] = 0
    w.w_packed = oracle.pack(codes)
    x = np.zeros((3, K), np.uint16)
    x[1, 5] = 0x3F80
    x[2, 7] = 0x7FC0  # NaN
    got = run(dev, x, w)
    assert not got[0].any()
    assert np.array_equal(got[1], w.biases[:, 0])
    assert np.all((got[2] & 0x7F80) == 0x7F80) and np.all(got[2] & 0x007F)


# ---------------------------------------------------------------- TMA-fed kernel (M <= 8, K % 512 == 0)

@pytest.mark.parametrize("M,N,K", [
    (1, 1, 512), (1, 16, 512), (1, 17, 1024), (1, 33, 2560), (1, 100, 4096), (1, 257, 14336), (1, 64, 16384),
    (2, 45, 1536), (2, 300, 8192), (3, 31, 3072), (4, 200, 4096), (5, 15, 2048), (8, 77, 2048), (7, 129, 512),
    (2, 50, 8704), (8, 40, 2560),   # M*K beyond the TMA kernel's x budget: generic kernel
])
def test_tma_kernel_shapes(dev, M, N, K):
    check(dev, M, N, K, 7 * M + N + K)


def test_tma_kernel_many_tiles_per_cta(dev):
    # more 32-row tiles than CTAs (two per SM): every CTA walks several tiles and stages wrap the ring
    check(dev, 1, 32 * 304 * 3 + 5, 1024, 77)


@pytest.mark.parametrize("M", [1, 4])
def test_tma_kernel_x_dynamic_range(dev, M):
    """Rows of x scaled by 2^-100, 2^100 and into the bf16 subnormal range, and a
    row mixing magnitudes 2^20 apart: the kernel stages each row of x in fp16
    with its own power-of-two scale, which keeps every element exact.  Each
    output row is checked against the oracle with that row's own RMS."""
    import torch
    N, K = 96, 2048
    w = synth.make_weights(N, K, 31)
    base = bf16_to_f64(synth.make_x(4, K, 31))
    base[0] *= 2.0 ** -100
    base[1] *= 2.0 ** 100
    base[2, ::3] *= 2.0 ** -20
    base[3] *= 2.0 ** -128
    x = synth.f32_to_bf16_bits(base.astype(np.float32))
    rows = [x[i:i + 1] for i in range(4)] if M == 1 else [x]
    for xr in rows:
        got = run(dev, xr, w)
        _, ref = oracle.matmul(xr, w.w_packed, w.scales, w.biases, xr.shape[0], N, K)
        for m in range(xr.shape[0]):
            assert_parity(got[m], ref[m], what=f"row {m} of {xr.shape[0]}")


def test_bounded_wait_timeout_reports_status(dev):
    """The test hook leaves out the first stage's copy: the consumers' bounded
    wait expires, the kernel records a timeout, the host reads AQ_ERR_TIMEOUT,
    and the context stays usable (a normal call right after is correct)."""
    import torch
    M, N, K = 1, 64, 1024
    w = synth.make_weights(N, K, 8)
    x = synth.make_x(M, K, 8)
    xt, wt, st, bt = upload(x, w, dev)
    assert aq.aq_read_device_status(None) == aq.AQ_OK
    aq.matmul(xt, wt, st, bt, flags=aq.AQ_FLAG_DEBUG_SKIP_COPY)
    assert aq.aq_read_device_status(torch.cuda.current_stream().cuda_stream) == aq.AQ_ERR_TIMEOUT
    assert aq.aq_read_device_status(None) == aq.AQ_OK          # cleared by the read
    check(dev, M, N, K, 8)
    with pytest.raises(aq.AqError):
        aq.matmul(xt[:, :64].contiguous(), wt[:, :8].contiguous(), st[:, :1].contiguous(), bt[:, :1].contiguous(),
                  flags=aq.AQ_FLAG_DEBUG_SKIP_COPY)                # K = 64: no TMA kernel, hook unsupported


# ---------------------------------------------------------------- 8-bit codes (TMA-fed kernel)

@pytest.mark.parametrize("M,N,K", [
    (1, 1, 512), (1, 33, 1024), (1, 100, 4096), (1, 4096, 4096), (1, 14336, 4096), (1, 4096, 14336),
    (1, 64, 16384), (2, 300, 2048), (3, 31, 3072), (8, 77, 2048), (5, 129, 1024), (7, 40, 1536),
    (16, 64, 1024), (4, 50, 8704), (20, 96, 512),   # rows beyond one staged pass: several launches
])
def test_eight_bit_shapes(dev, M, N, K):
    check(dev, M, N, K, 300 + M + N + K, bits=8)


def test_eight_bit_special_inputs(dev):
    """8-bit: zero x gives exact zeros, a one-hot x on a q = 0 column gives the
    bias, q = 255 gives 255*scale + bias, NaN propagates to its row."""
    N, K = 40, 1024
    w = synth.make_weights(N, K, 19, bits=8)
    codes = oracle.unpack(w.w_packed, N, K, 8)
    codes[:, 5] = 0
    codes[:, 700] = 255
    w.w_packed = oracle.pack(codes, 8)
    x = np.zeros((4, K), np.uint16)
    x[1, 5] = 0x3F80
    x[2, 700] = 0x3F80
    x[3, 7] = 0x7FC0  # NaN
    got = run(dev, x, w)
    _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, 4, N, K, bits=8)
    assert not got[0].any()
    assert np.array_equal(got[1], w.biases[:, 0])
    assert np.array_equal(got[2], ref[2])
    assert np.all((got[3] & 0x7F80) == 0x7F80) and np.all(got[3] & 0x007F)


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 64), (1, 100, 576), (2, 33, 1088), (3, 300, 4160), (8, 64, 14400), (9, 77, 576), (16, 40, 640),
    (20, 129, 1088), (40, 65, 192),
])
def test_eight_bit_general_kernel(dev, M, N, K):
    """8-bit codes with K not a multiple of 512: the general decode kernel (each
    code pair through the MMA as its two nibbles), in launches of 16 rows of x
    for any M, against the oracle; the explicit tensor-core choice is refused."""
    check(dev, M, N, K, 1700 + M + N + K, bits=8, kernel="auto")
    check(dev, M, N, K, 1800 + M + N + K, bits=8, kernel="qmv")
    if M > 16:
        w = synth.make_weights(N, K, 1, bits=8)
        xt, wt, st, bt = upload(synth.make_x(M, K, 1), w, dev)
        with pytest.raises(aq.AqError):
            aq.matmul(xt, wt, st, bt, bits=8, kernel="qmm")


def test_eight_bit_general_kernel_endpoints(dev):
    """The general kernel's 8-bit fold: a one-hot x over a q = 0 column gives
    the bias exactly (|bias| well above |scale| / 16 here, so the fold's fp32
    rounding stays below half a bf16 ulp), and q = 255, 15, 16, 240 (both
    nibbles, one nibble set) give scale * q + bias within the usual bound."""
    N, K = 45, 576
    w = synth.make_weights(N, K, 29, bits=8)
    codes = oracle.unpack(w.w_packed, N, K, 8)
    for col, q in ((3, 0), (100, 255), (200, 15), (300, 16), (575, 240)):
        codes[:, col] = q
    w.w_packed = oracle.pack(codes, 8)
    x = np.zeros((5, K), np.uint16)
    for r, col in enumerate((3, 100, 200, 300, 575)):
        x[r, col] = 0x3F80
    got = run(dev, x, w, kernel="qmv")
    _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, 5, N, K, bits=8)
    assert np.array_equal(got[0], w.biases[:, 0])
    assert_parity(got, ref, what="8-bit general kernel endpoints")


def test_eight_bit_rejected_where_unsupported(dev):
    import torch
    w = synth.make_weights(8, 512, 1, bits=8)
    x = synth.make_x(32, 512, 1)
    xt, wt, st, bt = upload(x, w, dev)
    # scales 2 bytes past a 16-byte boundary: neither 8-bit kernel can load them
    flat = torch.empty(st.numel() + 1, dtype=st.dtype, device=st.device)
    st_off = flat[1:].view(st.shape)
    st_off.copy_(st)
    with pytest.raises(aq.AqError):
        aq.matmul(xt, wt, st_off, bt, bits=8, kernel="qmm")
    with pytest.raises(aq.AqError):
        aq.matmul(xt[:1].contiguous(), wt, st_off, bt, bits=8)
    torch.cuda.synchronize()


def test_read_probe_streams_a_buffer(dev):
    """The read-only stream probe reads a buffer (a ragged number of chunks per
    SM, plus a tail shorter than a chunk that it leaves out) and leaves the
    device status clean."""
    import torch
    buf = torch.zeros((64 << 20) + 5 * 16384 + 100, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        assert aq.aq_read_probe(buf.data_ptr(), buf.numel(), stream) == aq.AQ_OK
    assert aq.aq_read_device_status(stream) == aq.AQ_OK
    assert int(buf.sum()) == 0
