"""CPU tests of the C ABI: the library loads, exports what include/aq.h
declares, rejects bad arguments before touching a device, and its host
utilities agree bit for bit with the oracle's."""
import ctypes

import numpy as np
import pytest

import affine_bit_quantized_gb300 as aq
import oracle
from affine_bit_quantized_gb300 import _build

A = 0x10000  # a 64 KiB-aligned fake address: validation never dereferences it


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build_library()


def test_exports_every_declared_symbol():
    names = aq.declared_functions()
    assert {"aq_matmul_bf16", "aq_matmul_bf16_ex", "aq_quantize_ref", "aq_pack_ref", "aq_status_string",
            "aq_last_cuda_error"} <= set(names)
    lib = ctypes.CDLL(aq.library_path())
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    for code, name in ((0, "AQ_OK"), (1, "AQ_ERR_INVALID_ARG"), (2, "AQ_ERR_UNSUPPORTED"), (3, "AQ_ERR_ALIGNMENT"),
                       (4, "AQ_ERR_CUDA"), (5, "AQ_ERR_TIMEOUT"), (6, "AQ_ERR_BAD_INDEX")):
        assert aq.status_string(code) == name
    assert aq.last_cuda_error() == ""


@pytest.mark.parametrize("args,expect", [
    (dict(bits=3), aq.AQ_ERR_UNSUPPORTED),
    (dict(bits=8, s=A + 2), aq.AQ_ERR_ALIGNMENT),    # 8-bit codes need 16-byte aligned scales
    (dict(bits=8, K=1024, b=A + 8), aq.AQ_ERR_ALIGNMENT),  # ... and biases
    (dict(group_size=32), aq.AQ_ERR_UNSUPPORTED),
    (dict(group_size=128), aq.AQ_ERR_UNSUPPORTED),
    (dict(K=96), aq.AQ_ERR_INVALID_ARG),
    (dict(M=-1), aq.AQ_ERR_INVALID_ARG),
    (dict(N=-5), aq.AQ_ERR_INVALID_ARG),
    (dict(K=-64), aq.AQ_ERR_INVALID_ARG),
    (dict(x=None), aq.AQ_ERR_INVALID_ARG),
    (dict(w=None), aq.AQ_ERR_INVALID_ARG),
    (dict(s=None), aq.AQ_ERR_INVALID_ARG),
    (dict(b=None), aq.AQ_ERR_INVALID_ARG),
    (dict(y=None), aq.AQ_ERR_INVALID_ARG),
    (dict(x=A + 8), aq.AQ_ERR_ALIGNMENT),
    (dict(w=A + 4), aq.AQ_ERR_ALIGNMENT),
    (dict(s=A + 1), aq.AQ_ERR_ALIGNMENT),
    (dict(b=A + 1), aq.AQ_ERR_ALIGNMENT),
    (dict(y=A + 1), aq.AQ_ERR_ALIGNMENT),
    (dict(M=0), aq.AQ_OK),          # empty: nothing launched
    (dict(N=0), aq.AQ_OK),
    (dict(M=0, x=None, y=None), aq.AQ_OK),
    (dict(M=1 << 31), aq.AQ_ERR_INVALID_ARG),
])
def test_validation_before_launch(args, expect):
    p = dict(x=A, w=A, s=A, b=A, y=A, M=1, N=64, K=128, group_size=64, bits=4)
    p.update(args)
    st = aq.aq_matmul_bf16(p["x"], p["w"], p["s"], p["b"], p["y"], p["M"], p["N"], p["K"], p["group_size"],
                           p["bits"], None)
    assert st == expect, aq.status_string(st)


def test_ex_rejects_unknown_kernel_and_flags():
    assert aq.aq_matmul_bf16_ex(A, A, A, A, A, 1, 64, 128, 64, 4, 7, 0, None) == aq.AQ_ERR_INVALID_ARG
    # 8-bit codes on the tensor-core kernel need K % 512 == 0: refused before any launch
    assert aq.aq_matmul_bf16_ex(A, A, A, A, A, 64, 64, 576, 64, 8, aq.AQ_KERNEL_QMM, 0, None) == aq.AQ_ERR_UNSUPPORTED
    assert aq.aq_matmul_bf16_ex(A, A, A, A, A, 1, 64, 128, 64, 4, 0, 1 << 5, None) == aq.AQ_ERR_INVALID_ARG
    assert aq.aq_matmul_bf16_ex(A, A, A, A, A, 0, 64, 128, 64, 4, 2, 1, None) == aq.AQ_OK


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_ref_matches_oracle(bits):
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 1 << bits, size=(9, 256), dtype=np.uint8)
    assert np.array_equal(aq.pack_ref(codes, bits), oracle.pack(codes, bits))


def test_pack_ref_rejects_out_of_range_code():
    codes = np.zeros((1, 8), np.uint8)
    codes[0, 3] = 16
    out = np.zeros((1, 1), np.uint32)
    assert aq.aq_pack_ref(codes.ctypes.data, 1, 8, 4, out.ctypes.data) == aq.AQ_ERR_INVALID_ARG


@pytest.mark.parametrize("bits", [4, 8])
def test_quantize_ref_matches_oracle(bits):
    rng = np.random.default_rng(8)
    w = rng.normal(0, 0.03, size=(17, 512)).astype(np.float32)
    w[3, :64] = -0.5                                  # constant group
    w[4, 64:128] = rng.normal(0, 1e-30, 64)           # tiny values: subnormal-range rounding
    w[5, 128:192] *= 1e4
    got = aq.quantize_ref(w, bits=bits)
    want = oracle.quantize(w, bits=bits)
    for g, o in zip(got, want):
        assert np.array_equal(g, o)


def _desc(**kw):
    d = dict(x=A, w_packed=A, scales=A, biases=A, y=A, M=1, N=64, K=512, flags=0)
    d.update(kw)
    return aq.MatmulDesc(d["x"], d["w_packed"], d["scales"], d["biases"], d["y"], d["M"], d["N"], d["K"], d["flags"])


@pytest.mark.parametrize("kw,expect", [
    (dict(M=9), aq.AQ_ERR_UNSUPPORTED),
    (dict(K=576), aq.AQ_ERR_UNSUPPORTED),        # not a multiple of 512
    (dict(K=96), aq.AQ_ERR_INVALID_ARG),
    (dict(M=2, K=16384), aq.AQ_ERR_UNSUPPORTED), # M*K beyond the staged-x limit
    (dict(N=0), aq.AQ_ERR_INVALID_ARG),
    (dict(x=None), aq.AQ_ERR_INVALID_ARG),
    (dict(x=A + 8), aq.AQ_ERR_ALIGNMENT),
    (dict(scales=A + 2), aq.AQ_ERR_ALIGNMENT),
])
def test_chain_prepare_validation(kw, expect):
    arr = (aq.MatmulDesc * 2)(_desc(), _desc(**kw))
    plan = aq.ChainPlan()
    nbytes = aq.aq_chain_workspace_bytes(2)
    assert aq.aq_chain_prepare(arr, 2, 64, 4, A, nbytes, plan) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(K=256 + 16), aq.AQ_ERR_UNSUPPORTED),    # not a multiple of 256
    (dict(K=40), aq.AQ_ERR_INVALID_ARG),          # not a multiple of 16
    (dict(M=9), aq.AQ_ERR_UNSUPPORTED),
    (dict(M=2, K=8192 + 256), aq.AQ_ERR_UNSUPPORTED),   # K rounds up to 10240: M*K beyond the staged-x limit
    (dict(biases=A + 2), aq.AQ_ERR_ALIGNMENT),    # the global scale: 4-byte aligned
    (dict(scales=A + 8), aq.AQ_ERR_ALIGNMENT),
    (dict(biases=None), aq.AQ_ERR_INVALID_ARG),
])
def test_chain_prepare_validation_nvfp4(kw, expect):
    """NVFP4 chains (group size 16, 4-bit): K a multiple of 256, scales 16-byte
    aligned, `biases` the 4-byte aligned address of the global scale."""
    arr = (aq.MatmulDesc * 2)(_desc(K=1024, biases=A + 4), _desc(**{"K": 1024, **kw}))
    plan = aq.ChainPlan()
    nbytes = aq.aq_chain_workspace_bytes(2)
    assert aq.aq_chain_prepare(arr, 2, 16, 4, A, nbytes, plan) == expect
    assert aq.aq_chain_prepare(arr, 2, 16, 8, A, nbytes, plan) == aq.AQ_ERR_UNSUPPORTED   # NVFP4 is 4-bit
    assert aq.aq_chain_prepare(arr, 2, 32, 4, A, nbytes, plan) == aq.AQ_ERR_UNSUPPORTED


def test_chain_workspace_and_plan_checks():
    assert aq.aq_chain_workspace_bytes(0) == 0
    assert aq.aq_chain_workspace_bytes(225) == 225 * 512 + 1024
    arr = (aq.MatmulDesc * 1)(_desc())
    plan = aq.ChainPlan()
    assert aq.aq_chain_prepare(arr, 1, 64, 4, A, 100, plan) == aq.AQ_ERR_INVALID_ARG      # workspace too small
    assert aq.aq_chain_prepare(arr, 1, 64, 4, A + 64, 4096, plan) == aq.AQ_ERR_ALIGNMENT   # not 128-aligned
    assert aq.aq_chain_prepare(arr, 1, 64, 2, A, 4096, plan) == aq.AQ_ERR_UNSUPPORTED
    assert aq.aq_chain_prepare(arr, 0, 64, 4, None, 0, plan) == aq.AQ_OK and plan.count == 0
    assert aq.aq_chain_run(plan, None) == aq.AQ_OK                                          # empty chain


@pytest.mark.parametrize("flags", [4, 0x10000000, 1 << 40])
def test_chain_prepare_rejects_unknown_flags(flags):
    # bits other than AQ_CHAIN_INDEPENDENT, AQ_CHAIN_RELEASE and the test hook, the
    # library's own record bit included
    arr = (aq.MatmulDesc * 1)(_desc(flags=flags))
    plan = aq.ChainPlan()
    assert aq.aq_chain_prepare(arr, 1, 64, 4, A, aq.aq_chain_workspace_bytes(1), plan) == aq.AQ_ERR_INVALID_ARG


# ---------------------------------------------------------------- expert-indexed matmul: validation

def _gather_call(**kw):
    d = dict(x=A, w=A, s=A, b=A, lhs=A, rhs=A, y=A, R=64, T=32, N=256, K=512, E=4, group_size=64, bits=4,
             ws=A, ws_bytes=None)
    d.update(kw)
    if d["ws_bytes"] is None:
        d["ws_bytes"] = aq.aq_gather_qmm_workspace_bytes(d["R"], d["K"], d["E"])
    return aq.aq_gather_qmm_bf16(d["x"], d["w"], d["s"], d["b"], d["lhs"], d["rhs"], d["y"], d["R"], d["T"], d["N"],
                                 d["K"], d["E"], d["group_size"], d["bits"], d["ws"], d["ws_bytes"], None)


def test_gather_workspace_bytes():
    # plan header (128) + one 16-byte tile per 128 rows plus one per expert, rounded to 128, then R*K*2
    assert aq.aq_gather_qmm_workspace_bytes(4096, 4096, 8) == 128 * ((128 + 16 * (32 + 8) + 127) // 128) + 4096 * 4096 * 2
    assert aq.aq_gather_qmm_workspace_bytes(0, 4096, 8) == 128 * ((128 + 16 * 8 + 127) // 128)
    assert aq.aq_gather_qmm_workspace_bytes(1, 512, 2000) == 0          # more experts than supported


@pytest.mark.parametrize("kw,expect", [
    (dict(bits=3), aq.AQ_ERR_UNSUPPORTED),
    (dict(group_size=32), aq.AQ_ERR_UNSUPPORTED),
    (dict(K=576), aq.AQ_ERR_UNSUPPORTED),          # not a multiple of 512 (the tensor-core K step)
    (dict(K=100), aq.AQ_ERR_INVALID_ARG),          # not a multiple of the group size
    (dict(E=0), aq.AQ_ERR_INVALID_ARG),
    (dict(E=1025), aq.AQ_ERR_INVALID_ARG),
    (dict(T=0), aq.AQ_ERR_INVALID_ARG),
    (dict(R=-1), aq.AQ_ERR_INVALID_ARG),
    (dict(lhs=None), aq.AQ_ERR_INVALID_ARG),
    (dict(ws=None), aq.AQ_ERR_INVALID_ARG),
    (dict(ws_bytes=1000), aq.AQ_ERR_INVALID_ARG),  # workspace too small
    (dict(x=A + 8), aq.AQ_ERR_ALIGNMENT),
    (dict(s=A + 2), aq.AQ_ERR_ALIGNMENT),
    (dict(rhs=A + 2), aq.AQ_ERR_ALIGNMENT),
    (dict(ws=A + 64), aq.AQ_ERR_ALIGNMENT),
    (dict(R=0, x=None, y=None), aq.AQ_OK),         # no rows: nothing launched
])
def test_gather_validation(kw, expect):
    assert _gather_call(**kw) == expect


# ---------------------------------------------------------------- NVFP4 matmul: validation

@pytest.mark.parametrize("kw,expect", [
    (dict(K=100), aq.AQ_ERR_INVALID_ARG),          # not a multiple of 16
    (dict(K=272), aq.AQ_ERR_UNSUPPORTED),          # not a multiple of 256
    (dict(K=32768 + 256), aq.AQ_ERR_UNSUPPORTED),  # one row of x beyond the 64 KB staging room
    (dict(M=-1), aq.AQ_ERR_INVALID_ARG),
    (dict(flags=1 << 3), aq.AQ_ERR_INVALID_ARG),
    (dict(x=None), aq.AQ_ERR_INVALID_ARG),
    (dict(x=A + 8), aq.AQ_ERR_ALIGNMENT),
    (dict(s=A + 4), aq.AQ_ERR_ALIGNMENT),
    (dict(M=0, x=None), aq.AQ_OK),
    (dict(N=0), aq.AQ_OK),
])
def test_nvfp4_validation(kw, expect):
    d = dict(x=A, w=A, s=A, g=1.0, y=A, M=1, N=64, K=512, flags=0)
    d.update(kw)
    assert aq.aq_matmul_nvfp4_bf16(d["x"], d["w"], d["s"], d["g"], d["y"], d["M"], d["N"], d["K"], d["flags"],
                                   None) == expect


# ---------------------------------------------------------------- workspace variant: validation

def test_matmul_workspace_bytes():
    assert aq.aq_matmul_workspace_bytes(16, 4096) == 0          # decode path: no workspace used
    assert aq.aq_matmul_workspace_bytes(17, 512) == 17 * 512 * 2
    assert aq.aq_matmul_workspace_bytes(2048, 4096) == 2048 * 4096 * 2
    assert aq.aq_matmul_workspace_bytes(-1, 4096) == 0


@pytest.mark.parametrize("args", [dict(bits=3), dict(group_size=32), dict(K=96), dict(x=A + 8), dict(M=-1),
                                  dict(x=None)])
def test_ws_variant_rejects_like_the_plain_call(args):
    p = dict(x=A, w=A, s=A, b=A, y=A, M=64, N=64, K=128, group_size=64, bits=4)
    p.update(args)
    plain = aq.aq_matmul_bf16(p["x"], p["w"], p["s"], p["b"], p["y"], p["M"], p["N"], p["K"], p["group_size"],
                              p["bits"], None)
    ws = aq.aq_matmul_bf16_ws(p["x"], p["w"], p["s"], p["b"], p["y"], p["M"], p["N"], p["K"], p["group_size"],
                              p["bits"], A, 1 << 20, None)
    assert plain != aq.AQ_OK and ws == plain


def test_read_probe_validation():
    """The read probe checks its arguments before any CUDA call."""
    assert aq.aq_read_probe(None, 1 << 20, None) == aq.AQ_ERR_INVALID_ARG
    assert aq.aq_read_probe(0x10000, 16383, None) == aq.AQ_ERR_INVALID_ARG
    assert aq.aq_read_probe(0x10008, 1 << 20, None) == aq.AQ_ERR_ALIGNMENT
