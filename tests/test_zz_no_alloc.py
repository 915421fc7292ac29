"""The allocation-free chain entry point (aq_chain_run_static).

Some callers cannot give this library device memory: a plugin inside a host
framework that owns the whole device memory pool and exposes no workspace, or
a serving loop that must not call an allocator after start-up.  For them
aq_chain_run_static keeps the chain's plan and completion counters in a
static device array.  These tests call it through the C ABI and check that it
gives exactly the bits of the workspace-based aq_chain_run (the same kernel in
the same order, so bit-equality is the right bar; it implies the parity
tolerance used everywhere else):
  * two calls in a row of one chain, with new inputs in between;
  * then a call with other weight buffers and other shapes, so that a record
    or tensor map left over from the previous call would show;
  * 8-bit codes, NVFP4 weights, and chains with several rows of x.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

import affine_bit_quantized_gb300 as aq
from affine_bit_quantized_gb300 import _build, synth

from ._helpers import to_dev_bf16, to_dev_u32, upload

A = 0x10000


def test_static_chain_rejects_more_than_its_scratch_holds():
    _build.build_library()
    arr = (aq.MatmulDesc * 257)()
    for i in range(257):
        arr[i] = aq.MatmulDesc(A, A, A, A, A, 1, 64, 512, 0)
    assert aq.aq_chain_run_static(arr, 257, 64, 4, None) == aq.AQ_ERR_INVALID_ARG
    assert aq.aq_chain_run_static(arr, 0, 64, 4, None) == aq.AQ_OK


def _layer_chain(dev, K, Ns, seed, M=1, bits=4, nvfp4=False):
    """q, k, v share xa; o reads q's output; gate, up share xm; down reads o's
    output.  Returns (items [(x, w, s, b, y, independent)], xa, xm); with
    nvfp4, s holds the E4M3 block scales and b the device fp32 tensor scale."""
    import torch
    nq, nk, nmlp, ndown = Ns
    plan = [("q", nq, K, "xa", 0), ("k", nk, K, "xa", 1), ("v", nk, K, "xa", 1), ("o", 2 * K, nq, "q", 0),
            ("gate", nmlp, K, "xm", 0), ("up", nmlp, K, "xm", 1), ("down", ndown, 2 * K, "o", 0)]
    xa = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    xm = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    outs, items = {}, []
    for i, (name, N, Kin, src, indep) in enumerate(plan):
        if nvfp4:
            w = synth.make_nvfp4_weights(N, Kin, seed + i)
            wt = to_dev_u32(w.w_packed, dev)
            st = torch.from_numpy(np.ascontiguousarray(w.scales)).to(dev)
            bt = torch.tensor([w.global_scale], dtype=torch.float32, device=dev)
        else:
            w = synth.make_weights(N, Kin, seed + i, bits=bits)
            wt, st, bt = upload(np.zeros((1, Kin), np.uint16), w, dev)[1:]
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        xin = {"xa": xa, "xm": xm}.get(src, outs.get(src))
        items.append((xin, wt, st, bt, y, indep))
        outs[name] = y
    return items, xa, xm


def _descs(items):
    return (aq.MatmulDesc * len(items))(*[
        aq.MatmulDesc(x.data_ptr(), w.data_ptr(), s.data_ptr(), b.data_ptr(), y.data_ptr(), x.shape[0], w.shape[0],
                      x.shape[1], aq.AQ_CHAIN_INDEPENDENT if ind else 0) for (x, w, s, b, y, ind) in items])


def _check_static_equals_workspace(dev, items, xa, xm, bits, calls, seed, group_size=64):
    """`calls` calls in a row, new inputs before each: the workspace chain
    first, then the static one on the same buffers; the outputs must be equal
    bit for bit."""
    import torch
    descs = _descs(items)
    ws_bytes = aq.aq_chain_workspace_bytes(len(items))
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    wplan = aq.ChainPlan()
    assert aq.aq_chain_prepare(descs, len(items), group_size, bits, workspace.data_ptr(), ws_bytes,
                               wplan) == aq.AQ_OK
    stream = torch.cuda.current_stream(dev).cuda_stream
    M, K = xa.shape
    for call in range(calls):
        xa.copy_(to_dev_bf16(synth.make_x(M, K, seed + 2 * call), dev))
        xm.copy_(to_dev_bf16(synth.make_x(M, K, seed + 2 * call + 1), dev))
        assert aq.aq_chain_run(wplan, stream) == aq.AQ_OK
        torch.cuda.synchronize()
        ref = [it[4].clone() for it in items]
        for it in items:
            it[4].fill_(float("nan"))
        assert aq.aq_chain_run_static(descs, len(items), group_size, bits, stream) == aq.AQ_OK
        torch.cuda.synchronize()
        assert aq.aq_read_device_status(stream) == aq.AQ_OK
        for i, (it, r) in enumerate(zip(items, ref)):
            assert torch.equal(it[4].view(torch.int16), r.view(torch.int16)), f"call {call} matmul {i}"


@pytest.mark.gpu
def test_static_chain_matches_workspace_chain_twice_then_on_other_buffers():
    import torch
    _build.build_library()
    dev = torch.device("cuda:0")
    items, xa, xm = _layer_chain(dev, 1024, (512, 128, 700, 1500), 300)
    _check_static_equals_workspace(dev, items, xa, xm, 4, calls=2, seed=400)
    # other weight buffers, other shapes: the records and tensor maps in the
    # static array are all replaced
    items2, xa2, xm2 = _layer_chain(dev, 2048, (1024, 256, 3000, 777), 350)
    _check_static_equals_workspace(dev, items2, xa2, xm2, 4, calls=1, seed=450)


@pytest.mark.gpu
@pytest.mark.parametrize("M,bits", [(1, 8), (3, 4), (2, 8)])
def test_static_chain_eight_bit_and_several_rows(M, bits):
    import torch
    _build.build_library()
    dev = torch.device("cuda:0")
    items, xa, xm = _layer_chain(dev, 1024, (512, 128, 700, 300), 600 + 10 * M + bits, M=M, bits=bits)
    _check_static_equals_workspace(dev, items, xa, xm, bits, calls=2, seed=700 + M)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 2])
def test_static_chain_nvfp4(M):
    """NVFP4 weights through the static entry point (group size 16): the same
    bits as the workspace chain, twice in a row."""
    import torch
    _build.build_library()
    dev = torch.device("cuda:0")
    items, xa, xm = _layer_chain(dev, 1024, (512, 128, 768, 300), 800 + M, M=M, nvfp4=True)
    _check_static_equals_workspace(dev, items, xa, xm, 4, calls=2, seed=900 + M, group_size=16)
