"""The benchmark's host-side arithmetic and its reference arm, on the CPU.

The algorithmic byte count is pinned to the storage format (4-bit codes plus
a bf16 scale and a bf16 bias per group of 64: 0.5625 bytes per weight; 8-bit
codes: 1.0625) and to the llama-3.1-8B shapes the workload stands in for; the
reference arm's JSON line is checked key by key.  No GPU is touched."""
import argparse
import contextlib
import io
import json
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("N,K", [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336), (128256, 4096)])
def test_alg_bytes_per_weight(N, K):
    act = 2 * K + 2 * N   # one bf16 row of x in, one bf16 row of y out
    assert (bench.alg_bytes(1, N, K) - act) * 16 == N * K * 9            # 0.5625 B per weight
    assert (bench.alg_bytes(1, N, K, bits=8) - act) * 16 == N * K * 17   # 1.0625 B per weight
    assert bench.alg_bytes(4, N, K) - bench.alg_bytes(1, N, K) == 3 * act


def test_step_is_the_8b_decode_step():
    mats = bench.step_matrices(32)
    assert len(mats) == 32 * 7 + 1
    layer = [(name, N, K) for (l, _, name, N, K, _) in mats if l == 0]
    assert layer == [("q_proj", 4096, 4096), ("k_proj", 1024, 4096), ("v_proj", 1024, 4096),
                     ("o_proj", 4096, 4096), ("gate_proj", 14336, 4096), ("up_proj", 14336, 4096),
                     ("down_proj", 4096, 14336)]
    assert sum(N * K for (_, N, K) in layer) // 2 == 109_051_904          # 4-bit codes of one layer
    assert mats[-1][2:5] == ("lm_head", 128256, 4096)
    assert 128256 * 4096 // 2 == 262_668_288                               # lm_head codes
    # every matrix of the step has its own seed: no weight copy is read twice per step
    assert len({m[5] for m in mats}) == len(mats)


def test_step_bytes_match_the_committed_traffic_summary():
    """The committed ncu summary scales its 4-layer capture by the same
    algorithmic bytes that the benchmark divides by."""
    text = open(os.path.join(ROOT, "profiles", "qmv_chain_decode_step_dram_traffic.txt")).read()

    def figure(pattern):
        return int(re.search(pattern, text).group(1).replace(",", ""))

    four = sum(bench.alg_bytes(1, N, K) for (_, _, _, N, K, _) in bench.step_matrices(4))
    full = sum(bench.alg_bytes(1, N, K) for (_, _, _, N, K, _) in bench.step_matrices(32))
    assert figure(r"algorithmic bytes ([\d,]+)") == four
    assert figure(r"full step: algorithmic ([\d,]+)") == full
    ratio = float(re.search(r"ratio ([\d.]+)", text).group(1))
    assert abs(figure(r"dram_bytes_per_step: (\d+)") - full * ratio) < 1e-4 * full


def test_x_layout_is_contiguous_per_role():
    offs, total = bench.x_layout(2)
    spans = sorted((o, K) for (o, K, _) in offs.values())
    pos = 0
    for o, K in spans:
        assert o == pos
        pos += K
    assert pos == total == 2 * (3 * 4096 + 14336) + 4096


def test_job_rate_is_weak_scaling():
    assert bench.job_rate(1, 4.0e9, 1e-3) == pytest.approx(4.0e12)
    assert bench.job_rate(8, 4.0e9, 1e-3) == pytest.approx(8 * 4.0e12)


def test_reference_arm_line():
    args = argparse.Namespace(steps=2, warmup=3, gpus=1)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, target_seconds=1.0)
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_side_measurements_above_every_ceiling_are_refused():
    """A side measurement far above the device's ceilings timed no work (a
    graph capture that recorded nothing): the benchmark refuses to print it."""
    ok_moe = {"w1_gate": {"us_per_call": 450.0, "tflops": 1068.7}}
    bad_moe = {"w1_gate": {"us_per_call": 0.73, "tflops": 659315.1}}
    per_matrix = {"lm_head": {"us_per_call": 49.4, "gbs": 5985.0}}
    bench.check_side_rates(per_matrix, None, None, None, None, ok_moe, 7450.0, 1915.6)
    with pytest.raises(RuntimeError, match="no work timed"):
        bench.check_side_rates(per_matrix, None, None, None, None, bad_moe, 7450.0, 1915.6)
    with pytest.raises(RuntimeError, match="lm_head"):
        bench.check_side_rates({"lm_head": {"gbs": 60000.0}}, None, None, None, None, None, 7450.0, 1915.6)
