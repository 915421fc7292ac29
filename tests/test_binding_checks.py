"""The Python binding's operand checks, on CPU tensors.

The C ABI receives bare pointers, so the binding checks every tensor's shape,
element type and placement before it calls the library; a tensor smaller than
(M, N, K) say would otherwise be read or written out of bounds on the device.
Shapes and types are checked before placement, so each case here reaches the
check it is about without a GPU; a call whose operands are all well formed
stops at "must be a contiguous CUDA tensor"."""
import pytest
import torch

import affine_bit_quantized_gb300 as aq

M, N, K = 2, 16, 128


def operands(bits=4, M=M, N=N, K=K):
    return dict(x=torch.zeros(M, K, dtype=torch.bfloat16),
                w_packed=torch.zeros(N, K * bits // 32, dtype=torch.int32),
                scales=torch.zeros(N, K // 64, dtype=torch.bfloat16),
                biases=torch.zeros(N, K // 64, dtype=torch.bfloat16))


def call_matmul(ops, **kw):
    return aq.matmul(ops["x"], ops["w_packed"], ops["scales"], ops["biases"], **kw)


@pytest.mark.parametrize("bits", [4, 8])
def test_well_formed_matmul_stops_at_placement(bits):
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        call_matmul(operands(bits), bits=bits)
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        call_matmul(operands(bits), bits=bits, out=torch.zeros(M, N, dtype=torch.bfloat16))


def test_uint32_codes_are_accepted():
    ops = operands()
    ops["w_packed"] = ops["w_packed"].view(torch.uint32)
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        call_matmul(ops)


@pytest.mark.parametrize("name,bad,match", [
    ("w_packed", torch.zeros(N, K // 8 - 1, dtype=torch.int32), "w_packed has shape"),
    ("w_packed", torch.zeros(N * K // 8, dtype=torch.int32), "x and w_packed must be 2-D"),
    ("w_packed", torch.zeros(N, K // 8, dtype=torch.float32), "w_packed has dtype"),
    ("w_packed", torch.zeros(N, K // 4, dtype=torch.int16), "w_packed has shape"),
    ("scales", torch.zeros(N, K // 64 - 1, dtype=torch.bfloat16), "scales has shape"),
    ("scales", torch.zeros(N - 1, K // 64, dtype=torch.bfloat16), "scales has shape"),
    ("scales", torch.zeros(N, K // 64, dtype=torch.float16), "scales has dtype"),
    ("biases", torch.zeros(N, K // 32, dtype=torch.bfloat16), "biases has shape"),
    ("biases", torch.zeros(N, K // 64, dtype=torch.float32), "biases has dtype"),
    ("x", torch.zeros(M, K, dtype=torch.float16), "x has dtype"),
    ("x", torch.zeros(M, K, 1, dtype=torch.bfloat16), "x and w_packed must be 2-D"),
])
def test_matmul_rejects_malformed_operand(name, bad, match):
    ops = operands()
    ops[name] = bad
    with pytest.raises(ValueError, match=match):
        call_matmul(ops)


def test_matmul_code_width_sets_the_word_count():
    with pytest.raises(ValueError, match="w_packed has shape"):
        call_matmul(operands(bits=4), bits=8)
    with pytest.raises(ValueError, match="w_packed has shape"):
        call_matmul(operands(bits=8), bits=4)


@pytest.mark.parametrize("out,match", [
    (torch.zeros(M, N + 1, dtype=torch.bfloat16), "out has shape"),
    (torch.zeros(M + 1, N, dtype=torch.bfloat16), "out has shape"),
    (torch.zeros(M * N, dtype=torch.bfloat16), "out has shape"),
    (torch.zeros(M, N, dtype=torch.float32), "out has dtype"),
])
def test_matmul_rejects_malformed_out(out, match):
    with pytest.raises(ValueError, match=match):
        call_matmul(operands(), out=out)


def test_matmul_workspace_and_kernel_checks():
    with pytest.raises(ValueError, match="workspace has dtype"):
        call_matmul(operands(), workspace=torch.zeros(64, dtype=torch.int32))
    with pytest.raises(ValueError, match="workspace has shape"):
        call_matmul(operands(), workspace=torch.zeros(8, 8, dtype=torch.uint8))
    with pytest.raises(ValueError, match="default kernel choice"):
        call_matmul(operands(), workspace=torch.zeros(64, dtype=torch.uint8), kernel="qmm")
    with pytest.raises(ValueError, match="kernel must be one of"):
        call_matmul(operands(), kernel="fast")


@pytest.mark.parametrize("K_,kw", [(96, {}), (K, {"bits": 3}), (K, {"group_size": 0})])
def test_shapes_the_library_rejects_are_left_to_it(K_, kw):
    # K not a multiple of the group, or an unsupported code width or group: the
    # word and group counts are not defined there, and the library's own status
    # (checked before any launch) answers instead
    ops = dict(x=torch.zeros(M, K_, dtype=torch.bfloat16), w_packed=torch.zeros(N, 12, dtype=torch.int32),
               scales=torch.zeros(N, 1, dtype=torch.bfloat16), biases=torch.zeros(N, 1, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        call_matmul(ops, **kw)


# ---------------------------------------------------------------- gather_qmm

E, T, R = 4, 6, 12


def gather_operands(bits=4):
    return dict(x=torch.zeros(T, K, dtype=torch.bfloat16),
                w_packed=torch.zeros(E, N, K * bits // 32, dtype=torch.int32),
                scales=torch.zeros(E, N, K // 64, dtype=torch.bfloat16),
                biases=torch.zeros(E, N, K // 64, dtype=torch.bfloat16),
                lhs_indices=torch.zeros(R, dtype=torch.int32),
                rhs_indices=torch.zeros(R, dtype=torch.int32))


@pytest.mark.parametrize("name,bad,match", [
    (None, None, "contiguous CUDA tensor"),
    ("w_packed", torch.zeros(E * N, K // 8, dtype=torch.int32), "w_packed 3-D"),
    ("w_packed", torch.zeros(E, N, K // 8 + 1, dtype=torch.int32), "w_packed has shape"),
    ("scales", torch.zeros(E - 1, N, K // 64, dtype=torch.bfloat16), "scales has shape"),
    ("biases", torch.zeros(E, N, K // 64, dtype=torch.float16), "biases has dtype"),
    ("rhs_indices", torch.zeros(R, dtype=torch.int64), "rhs_indices has dtype"),
    ("rhs_indices", torch.zeros(R - 1, dtype=torch.int32), "rhs_indices has shape"),
    ("lhs_indices", torch.zeros(R, dtype=torch.int64), "lhs_indices has dtype"),
    ("x", torch.zeros(T, K + 64, dtype=torch.bfloat16), "w_packed has shape"),
])
def test_gather_checks(name, bad, match):
    ops = gather_operands()
    if name is not None:
        ops[name] = bad
    with pytest.raises(ValueError, match=match):
        aq.gather_qmm(**ops)


def test_gather_out_and_workspace_checks():
    with pytest.raises(ValueError, match="out has shape"):
        aq.gather_qmm(**gather_operands(), out=torch.zeros(R, N + 1, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="workspace has dtype"):
        aq.gather_qmm(**gather_operands(), workspace=torch.zeros(16, dtype=torch.float32))
    with pytest.raises(ValueError, match="w_packed has shape"):
        aq.gather_qmm(**gather_operands(bits=4), bits=8)


# ---------------------------------------------------------------- NVFP4

@pytest.mark.parametrize("name,bad,match", [
    (None, None, "contiguous CUDA tensor"),
    ("w_packed", torch.zeros(N, K // 8 - 1, dtype=torch.int32), "w_packed has shape"),
    ("scales_e4m3", torch.zeros(N, K // 32, dtype=torch.uint8), "scales_e4m3 has shape"),
    ("scales_e4m3", torch.zeros(N, K // 16, dtype=torch.int8), "scales_e4m3 has dtype"),
    ("x", torch.zeros(M, K, dtype=torch.float32), "x has dtype"),
])
def test_nvfp4_checks(name, bad, match):
    ops = dict(x=torch.zeros(M, K, dtype=torch.bfloat16), w_packed=torch.zeros(N, K // 8, dtype=torch.int32),
               scales_e4m3=torch.zeros(N, K // 16, dtype=torch.uint8))
    if name is not None:
        ops[name] = bad
    with pytest.raises(ValueError, match=match):
        aq.matmul_nvfp4(ops["x"], ops["w_packed"], ops["scales_e4m3"], 1.0)


def test_nvfp4_out_check():
    with pytest.raises(ValueError, match="out has shape"):
        aq.matmul_nvfp4(torch.zeros(M, K, dtype=torch.bfloat16), torch.zeros(N, K // 8, dtype=torch.int32),
                        torch.zeros(N, K // 16, dtype=torch.uint8), 1.0, out=torch.zeros(N, M, dtype=torch.bfloat16))


# ---------------------------------------------------------------- chain

def test_chain_checks_every_item():
    a, b = operands(M=1), operands(M=1, N=K)   # b maps a row of K to K outputs
    y0 = torch.zeros(1, N, dtype=torch.bfloat16)
    y1 = torch.zeros(1, K, dtype=torch.bfloat16)
    good = [(a["x"], a["w_packed"], a["scales"], a["biases"], y1[:, :N].contiguous()),
            (b["x"], b["w_packed"], b["scales"], b["biases"], y1)]
    with pytest.raises(ValueError, match="chain item 0: x must be a contiguous CUDA tensor"):
        aq.Chain(good)
    bad = [good[0], (b["x"], b["w_packed"], b["scales"], b["biases"], y0)]
    with pytest.raises(ValueError, match="chain item 1: y has shape"):
        aq.Chain(bad)
    bad = [good[0], (b["x"], b["w_packed"], b["scales"][:, :1].contiguous(), b["biases"], y1)]
    with pytest.raises(ValueError, match="chain item 1: scales has shape"):
        aq.Chain(bad)


def test_chain_independent_flags_match_the_items():
    a = operands(M=1)
    item = (a["x"], a["w_packed"], a["scales"], a["biases"], torch.zeros(1, N, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="independent has 1 flags for 2 matmuls"):
        aq.Chain([item, item], independent=[False])


def test_static_chain_wrapper_checks_like_chain():
    a, b = operands(M=1), operands(M=1, N=K)
    y0 = torch.zeros(1, N, dtype=torch.bfloat16)
    y1 = torch.zeros(1, K, dtype=torch.bfloat16)
    good = [(a["x"], a["w_packed"], a["scales"], a["biases"], y1[:, :N].contiguous()),
            (b["x"], b["w_packed"], b["scales"], b["biases"], y1)]
    with pytest.raises(ValueError, match="chain item 0: x must be a contiguous CUDA tensor"):
        aq.chain_run_static(good)
    with pytest.raises(ValueError, match="chain item 1: y has shape"):
        aq.chain_run_static([good[0], (b["x"], b["w_packed"], b["scales"], b["biases"], y0)])
    with pytest.raises(ValueError, match="independent has 1 flags for 2 matmuls"):
        aq.chain_run_static(good, independent=[False])
