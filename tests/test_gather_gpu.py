"""GPU parity of the expert-indexed matmul (aq_gather_qmm_bf16, MoE prefill)
against the oracle, through the C ABI."""
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


def upload_experts(ew, dev):
    import torch
    w = to_dev_u32(ew.w_packed.reshape(ew.E * ew.N, -1), dev).view(ew.E, ew.N, -1)
    s = to_dev_bf16(ew.scales.reshape(ew.E * ew.N, -1), dev).view(ew.E, ew.N, -1)
    b = to_dev_bf16(ew.biases.reshape(ew.E * ew.N, -1), dev).view(ew.E, ew.N, -1)
    return w, s, b


def run(dev, x, ew, lhs, rhs, out=None):
    import torch
    w, s, b = upload_experts(ew, dev)
    xt = to_dev_bf16(x, dev)
    lt = torch.from_numpy(np.ascontiguousarray(lhs, np.int32)).to(dev)
    rt = torch.from_numpy(np.ascontiguousarray(rhs, np.int32)).to(dev)
    y = aq.gather_qmm(xt, w, s, b, lt, rt, out=out, bits=ew.bits)
    torch.cuda.synchronize()
    return y


def check(dev, T, E, N, K, top_k, seed, bits=4):
    ew = synth.ExpertWeights(E, N, K, seed, bits=bits)
    x = synth.make_x(T, K, seed)
    lhs, rhs = synth.make_routing(T, E, top_k, seed)
    got = from_dev_bf16(run(dev, x, ew, lhs, rhs))
    _, ref = oracle.gather_matmul(x, ew.w_packed, ew.scales, ew.biases, lhs, rhs, N, K, bits=bits)
    assert aq.aq_read_device_status(None) == aq.AQ_OK
    return assert_parity(got, ref, what=f"gather T={T} E={E} N={N} K={K} top{top_k} bits={bits}")


@pytest.mark.parametrize("T,E,N,K,top_k,bits", [
    (64, 4, 300, 1024, 2, 4),
    (64, 4, 300, 1024, 2, 8),
    (100, 8, 513, 1536, 2, 4),     # ragged N, segments of ~25 rows
    (600, 2, 256, 512, 1, 4),      # ~300 rows per expert: several row tiles per expert
    (300, 3, 700, 2048, 3, 8),     # every token to every expert
    (7, 16, 64, 512, 2, 4),        # most experts get one row or none
])
def test_gather_parity(dev, T, E, N, K, top_k, bits):
    check(dev, T, E, N, K, top_k, 700 + T + E + N, bits=bits)


def test_gather_empty_experts_and_arbitrary_rows(dev):
    """Experts 0 and 2 receive no rows, a token appears under several experts
    and a row pair repeats; every row still matches the oracle."""
    T, E, N, K = 40, 4, 260, 1024
    ew = synth.ExpertWeights(E, N, K, 11)
    x = synth.make_x(T, K, 11)
    lhs = np.array([3, 5, 5, 39, 0, 3, 3, 17, 17, 17], np.int32)
    rhs = np.array([1, 1, 1, 1, 3, 3, 3, 3, 3, 3], np.int32)
    got = from_dev_bf16(run(dev, x, ew, lhs, rhs))
    _, ref = oracle.gather_matmul(x, ew.w_packed, ew.scales, ew.biases, lhs, rhs, N, K)
    assert_parity(got, ref, what="gather empty experts")
    assert np.array_equal(got[1], got[2]) and np.array_equal(got[5], got[6])


def test_gather_deterministic(dev):
    import torch
    T, E, N, K = 256, 8, 512, 2048
    ew = synth.ExpertWeights(E, N, K, 12)
    x = synth.make_x(T, K, 12)
    lhs, rhs = synth.make_routing(T, E, 2, 12)
    a = run(dev, x, ew, lhs, rhs)
    b = run(dev, x, ew, lhs, rhs)
    assert torch.equal(a, b)


@pytest.mark.parametrize("bad", ["token", "expert", "order"])
def test_gather_bad_indices_reported_and_nothing_written(dev, bad):
    import torch
    T, E, N, K = 16, 4, 64, 512
    ew = synth.ExpertWeights(E, N, K, 13)
    x = synth.make_x(T, K, 13)
    lhs, rhs = synth.make_routing(T, E, 2, 13)
    lhs, rhs = lhs.copy(), rhs.copy()
    if bad == "token":
        lhs[5] = T
    elif bad == "expert":
        rhs[-1] = E
    else:
        rhs[0], rhs[-1] = rhs[-1], rhs[0]
    out = torch.full((lhs.size, N), float("nan"), dtype=torch.bfloat16, device=dev)
    run(dev, x, ew, lhs, rhs, out=out)
    assert aq.aq_read_device_status(None) == aq.AQ_ERR_BAD_INDEX
    assert torch.isnan(out.float()).all()
    assert aq.aq_read_device_status(None) == aq.AQ_OK          # cleared by the read
    check(dev, T, E, N, K, 2, 14)                               # the context stays usable


@pytest.mark.parametrize("j", [0, 2])
def test_gather_mixtral_shape_sampled(dev, j):
    """Mixtral-8x7B-shaped expert matrices (8 experts; 14336 x 4096, and the
    4096 x 14336 down projection, whose launch splits K across CTA pairs),
    2048 tokens routed top-2: sampled outputs (plus the last row and column)
    against the oracle."""
    T, E, (name, N, K), top_k = 2048, synth.MIXTRAL_EXPERTS, synth.MIXTRAL_EXPERT_MATS[j], synth.MIXTRAL_TOP_K
    ew = synth.ExpertWeights(E, N, K, synth.seed_for(6, j, 0))
    x = synth.make_x(T, K, synth.seed_for(6, j, 8))
    lhs, rhs = synth.make_routing(T, E, top_k, synth.seed_for(6, j, 9))
    got = from_dev_bf16(run(dev, x, ew, lhs, rhs))
    rng = np.random.default_rng(3)
    R = lhs.size
    ir = np.concatenate([rng.integers(0, R, 3000), [R - 1, 0, R - 1]])
    inn = np.concatenate([rng.integers(0, N, 3000), [N - 1, N - 1, 0]])
    ye, yb = oracle.gather_matmul_sampled(x, ew.w_packed, ew.scales, ew.biases, lhs, rhs, N, K, ir, inn)
    rms = float(np.sqrt(np.mean(ye * ye)))
    assert_parity(got[ir, inn], yb, rms=rms, what="mixtral gather sampled")


def test_gather_whole_waves_then_split_tail_8bit_sampled(dev):
    """8-bit expert matrices (4096 x 4096, 8 experts, 2048 tokens top-2): the
    row tiles that fill whole waves run in one launch, the remaining ones with
    K split across CTA pairs; sampled outputs (plus both ends of the last row
    tiles) against the oracle."""
    T, E, N, K, top_k = 2048, 8, 4096, 4096, 2
    ew = synth.ExpertWeights(E, N, K, 31, bits=8)
    x = synth.make_x(T, K, 32)
    lhs, rhs = synth.make_routing(T, E, top_k, 33)
    got = from_dev_bf16(run(dev, x, ew, lhs, rhs))
    rng = np.random.default_rng(5)
    R = lhs.size
    ir = np.concatenate([rng.integers(0, R, 3000), R - 1 - np.arange(64), [0, R - 1]])
    inn = np.concatenate([rng.integers(0, N, 3064), [N - 1, 0]])
    ye, yb = oracle.gather_matmul_sampled(x, ew.w_packed, ew.scales, ew.biases, lhs, rhs, N, K, ir, inn, bits=8)
    rms = float(np.sqrt(np.mean(ye * ye)))
    assert aq.aq_read_device_status(None) == aq.AQ_OK
    assert_parity(got[ir, inn], yb, rms=rms, what="gather 8-bit two launches sampled")
