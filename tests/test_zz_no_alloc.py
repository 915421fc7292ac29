"""The allocation-free chain entry point (aq_chain_run_static).

Some callers cannot give this library device memory: a plugin inside a host
framework that owns the whole device memory pool and exposes no workspace, or
a serving loop that must not call an allocator after start-up.  For them
aq_chain_run_static keeps the chain's plan and completion counters in a
static device array.  These tests check, through the C ABI, that two calls
in a row give the same results as the workspace-based aq_chain_run, within
the parity tolerance used everywhere else.  This file is collected last so
that a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

import affine_bit_quantized_gb300 as aq
from affine_bit_quantized_gb300 import _build, synth

from ._helpers import assert_parity, from_dev_bf16, to_dev_bf16, upload

A = 0x10000


def test_static_chain_rejects_more_than_its_scratch_holds():
    _build.build_library()
    arr = (aq.MatmulDesc * 257)()
    for i in range(257):
        arr[i] = aq.MatmulDesc(A, A, A, A, A, 1, 64, 512, 0)
    assert aq.aq_chain_run_static(arr, 257, 64, 4, None) == aq.AQ_ERR_INVALID_ARG
    assert aq.aq_chain_run_static(arr, 0, 64, 4, None) == aq.AQ_OK


@pytest.mark.gpu
def test_static_chain_matches_workspace_chain_twice():
    import torch
    _build.build_library()
    dev = torch.device("cuda:0")
    # a small decode-like chain: q, k, v share x; o reads q's output; gate, up
    # share a second x; down reads o's output
    K = 1024
    plan = [("q", 512, K, "xa", 0), ("k", 128, K, "xa", 1), ("v", 128, K, "xa", 1), ("o", 1024, 512, "q", 0),
            ("gate", 700, K, "xm", 0), ("up", 700, K, "xm", 1), ("down", 1500, 1024, "o", 0)]
    xa = torch.empty((1, K), dtype=torch.bfloat16, device=dev)
    xm = torch.empty((1, K), dtype=torch.bfloat16, device=dev)
    outs, items = {}, []
    for i, (name, N, Kin, src, indep) in enumerate(plan):
        w = synth.make_weights(N, Kin, 300 + i)
        wt, st, bt = upload(np.zeros((1, Kin), np.uint16), w, dev)[1:]
        y = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
        xin = {"xa": xa, "xm": xm}.get(src, outs.get(src))
        items.append((xin, wt, st, bt, y, indep))
        outs[name] = y
    descs = (aq.MatmulDesc * len(items))(*[
        aq.MatmulDesc(x.data_ptr(), w.data_ptr(), s.data_ptr(), b.data_ptr(), y.data_ptr(), x.shape[0], w.shape[0],
                      x.shape[1], aq.AQ_CHAIN_INDEPENDENT if ind else 0) for (x, w, s, b, y, ind) in items])
    ws_bytes = aq.aq_chain_workspace_bytes(len(items))
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    wplan = aq.ChainPlan()
    assert aq.aq_chain_prepare(descs, len(items), 64, 4, workspace.data_ptr(), ws_bytes, wplan) == aq.AQ_OK
    stream = torch.cuda.current_stream(dev).cuda_stream
    for call in range(2):                       # two calls in a row, with new inputs each time
        xa.copy_(to_dev_bf16(synth.make_x(1, K, 400 + call), dev))
        xm.copy_(to_dev_bf16(synth.make_x(1, K, 500 + call), dev))
        assert aq.aq_chain_run(wplan, stream) == aq.AQ_OK
        torch.cuda.synchronize()
        ref = [from_dev_bf16(it[4]) for it in items]
        for it in items:
            it[4].fill_(float("nan"))
        assert aq.aq_chain_run_static(descs, len(items), 64, 4, stream) == aq.AQ_OK
        torch.cuda.synchronize()
        assert aq.aq_read_device_status(stream) == aq.AQ_OK
        for (name, *_), it, r in zip(plan, items, ref):
            assert_parity(from_dev_bf16(it[4]), r, what=f"call {call} {name}")
