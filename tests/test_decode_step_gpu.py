"""The decode step the benchmark times, compared with the oracle.

The benchmark's headline number comes from one launch: the chained kernel
running a Llama-3.1-8B-shaped decode step (32 layers x q, k, v, o, gate, up,
down, plus lm_head; 225 matmuls, k, v and up flagged independent, lm_head
inside the chain).  This test builds that step with the module the benchmark
uses (same seeds, same buffers, same descriptors, same plan) and checks every
output of every matmul, element by element, against the plain fp64 definition
rounded once to bf16.  It also checks that the step is repeatable bit for bit
and that the graph of one launch per matmul (the benchmark's alternative)
gives the same bits as the chain.
"""
import numpy as np
import pytest

import oracle
from affine_bit_quantized_gb300 import _build, decode_step, synth

from ._helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def step():
    import torch
    _build.build_library()
    dev = torch.device("cuda:0")
    ds = decode_step.DecodeStep(dev, synth.LLAMA8B_LAYERS, keep_host=True)
    yield ds
    del ds
    torch.cuda.empty_cache()


def _host_y(ds) -> np.ndarray:
    return ds.y.cpu().numpy().view(np.uint16)


def test_step_layout_is_the_benchmarked_one(step):
    assert step.count == 32 * 7 + 1
    assert step.mats[-1][2] == "lm_head" and step.mats[-1][3:5] == (128256, 4096)
    assert sum(step.independent) == 32 * 3
    assert [m[2] for m, ind in zip(step.mats, step.independent) if ind] == ["k_proj", "v_proj", "up_proj"] * 32
    assert step.plan.count == step.count and step.plan.one_row == 1


def test_every_output_of_the_chained_step_matches_the_oracle(step):
    import torch
    import affine_bit_quantized_gb300 as aq

    step.y.fill_(0x7FC0)            # NaN bit pattern: an unwritten output fails
    stream = torch.cuda.current_stream(step.device)
    step.run_chain(stream.cuda_stream)
    torch.cuda.synchronize(step.device)
    assert aq.aq_read_device_status(stream.cuda_stream) == aq.AQ_OK
    y = _host_y(step)
    for i, (layer, j, name, N, K, seed) in enumerate(step.mats):
        w = step.host_weights[i]
        _, ref = oracle.matmul(step.host_x_row(i), w.w_packed, w.scales, w.biases, 1, N, K)
        got = y[step.y_offsets[i]:step.y_offsets[i] + N].reshape(1, N)
        assert_parity(got, ref, what=f"layer {layer} {name}")


def test_step_is_repeatable_and_equals_the_graph_of_single_launches(step):
    import torch

    stream = torch.cuda.current_stream(step.device)
    step.run_chain(stream.cuda_stream)
    torch.cuda.synchronize(step.device)
    first = step.y.clone()
    for _ in range(2):
        step.y.fill_(0x7FC0)
        step.run_chain(stream.cuda_stream)
    torch.cuda.synchronize(step.device)
    assert torch.equal(step.y, first)
    graph = step.capture_graph()
    step.y.fill_(0x7FC0)
    graph.replay()
    torch.cuda.synchronize(step.device)
    assert torch.equal(step.y, first)


def test_nvfp4_step_matches_the_oracle_and_single_launches():
    """The same step with NVFP4 weights (the benchmark's NVFP4 step line), on
    4 layers plus lm_head: every output of the chained launch against the
    NVFP4 oracle, and the same bits as one aq_matmul_nvfp4_bf16 per matmul
    (captured as a graph)."""
    import torch
    import affine_bit_quantized_gb300 as aq

    _build.build_library()
    dev = torch.device("cuda:0")
    ds = decode_step.DecodeStep(dev, 4, keep_host=True, fmt="nvfp4")
    assert ds.count == 4 * 7 + 1
    stream = torch.cuda.current_stream(dev)
    ds.y.fill_(0x7FC0)
    ds.run_chain(stream.cuda_stream)
    torch.cuda.synchronize(dev)
    assert aq.aq_read_device_status(stream.cuda_stream) == aq.AQ_OK
    y = _host_y(ds)
    for i, (layer, j, name, N, K, seed) in enumerate(ds.mats):
        w = ds.host_weights[i]
        _, ref = oracle.nvfp4_matmul(ds.host_x_row(i), w.w_packed, w.scales, w.global_scale, 1, N, K)
        got = y[ds.y_offsets[i]:ds.y_offsets[i] + N].reshape(1, N)
        assert_parity(got, ref, what=f"nvfp4 layer {layer} {name}")
    first = ds.y.clone()
    graph = ds.capture_graph()
    ds.y.fill_(0x7FC0)
    graph.replay()
    torch.cuda.synchronize(dev)
    assert torch.equal(ds.y, first)
