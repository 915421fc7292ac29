#!/usr/bin/env python
"""Benchmark: a Llama-3.1-8B-shaped decode step of the affine group-quantized matmul.

One step = every weight matrix of 32 decoder layers (q, k, v, o, gate, up,
down; 4-bit codes, group 64, bf16 scales and biases, each layer drawn from its
own seed) plus lm_head, each multiplied by one bf16 activation row (M = 1).
That is 4.22 GB of weights streamed per step, far larger than the 129 MB L2,
so consecutive steps never hit in L2.  The timed step is one cooperative
persistent launch of the chained decode kernel (aq_chain_run: matmul j reads
its x only after matmul j-1 has stored all of its y, except k, v and up, which
read the same x as the matmul before them); the same step as a CUDA graph of
one launch per matmul is reported beside it as "alt".

Prints one JSON line.  `value` is the achieved algorithmic HBM bandwidth of
the step in GB/s (bytes the definition must read and write: packed codes,
scales, biases, x and y), summed over ranks; `tok_s` is the equivalent decode
rate; the `qmm` object gives the prefill-sized tensor-core GEMM's TFLOPS on
the 4096x14336 / 14336x4096 shapes at M = 256 and 2048.

--impl reference times the CPU oracle (the plain fp64 definition) on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from affine_bit_quantized_gb300 import synth  # noqa: E402

METRIC = "qmv achieved HBM GB/s (% of GB300 peak) and 8B-shape equiv decode tok/s; qmm TFLOPS"
WORKLOAD = ("llama-3.1-8b-shaped decode step: 32 layers x (q,k,v,o,gate,up,down) + lm_head, "
            "M=1, 4-bit affine codes, group 64, bf16 scales/biases")
QMM_SHAPES = ((4096, 14336, "gate/up"), (14336, 4096, "down"))   # (K, N)
QMM_M = (256, 2048)


def alg_bytes(M: int, N: int, K: int, bits: int = 4) -> int:
    """Bytes the definition must move: codes (K*bits/8 per row), scales and
    biases (2 x 2 bytes per group of 64), x and y."""
    return N * K * bits // 8 + N * (K // 64) * 4 + 2 * M * K + 2 * M * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # wait (up to 10 s) for the first sample, so that nvidia-smi's start-up is
        # over before the timed region begins
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 10:
            self.file.flush()
            if os.path.getsize(self.file.name) > 0:
                break
            time.sleep(0.05)
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, power, reasons = [], [], [], set()
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload
# The step's layout (matrices, seeds, activation rows, independence flags) is
# shared with the tests that compare this exact launch with the oracle.
from affine_bit_quantized_gb300.decode_step import (  # noqa: E402
    CONFIG_ID, ROLE_OF, DecodeStep, step_matrices, x_layout)


def rank_env():
    """(world size, rank, local rank) from the launcher's environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(v: float, world: int, device) -> float:
    """The largest of every rank's v (a collective: every rank must call it)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, seconds_max: float) -> float:
    """Whole-job throughput of replicas (weak scaling): every rank processed
    units_per_rank, the slowest in seconds_max."""
    return world * units_per_rank / seconds_max


def run_reference(args, target_seconds: float = 150.0):
    """CPU oracle on a bounded sample of the decode step: the first R rows of
    each of the 7 matrices of one layer per step, R sized so that warm-up plus
    timed steps take about `target_seconds` on this host's cores."""
    import oracle

    mats = [m for m in step_matrices(1) if m[2] != "lm_head"]
    offs, _ = x_layout(1)
    full = []
    for (layer, j, name, N, K, seed) in mats:
        w = synth.make_weights(N, K, seed)
        full.append((synth.make_x(1, K, offs[(layer, ROLE_OF[name])][2]), w, N, K))
    threads = oracle.default_threads()

    def run_rows(R):
        for x, w, N, K in full:
            r = min(R, N)
            oracle.matmul(x, w.w_packed[:r], w.scales[:r], w.biases[:r], 1, r, K, nthreads=threads)

    t0 = time.perf_counter()
    run_rows(64)
    per_row = (time.perf_counter() - t0) / 64
    budget = target_seconds / (args.steps + args.warmup)
    R = int(max(8, min(1024, budget / max(per_row, 1e-9))))
    step_bytes = sum(alg_bytes(1, min(R, N), K) for (_, _, N, K) in full)
    for _ in range(args.warmup):
        run_rows(R)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_rows(R)
    dt = (time.perf_counter() - t0) / args.steps
    gbs = step_bytes / dt / 1e9
    sample = (f"first {R} rows of each of the 7 matrices of one 8B-shaped decode layer per step "
              f"({sum(min(R, N) * K for (_, _, N, K) in full) / 1e6:.1f} M weights), M=1, fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample, "M": 1},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_case(args):
    """Time y = x . dequant(W)^T for one (M, N, K) through the C ABI: enough
    distinct weight copies to exceed 3x L2 are cycled so that no launch finds
    its weights in L2; CUDA events around `steps` launches."""
    import torch

    import affine_bit_quantized_gb300 as aq
    from affine_bit_quantized_gb300 import _build

    M, N, K = (int(v) for v in args.case.split(","))
    bits = args.bits
    dev = torch.device("cuda", 0)
    _build.build_library()
    lib = aq.load()
    w = synth.make_weights(N, K, 1, bits=bits)
    x = synth.make_x(M, K, 1)
    wbytes = w.nbytes
    copies = max(1, min(64, -(-3 * 129 * 2**20 // wbytes)))
    ws = []
    for c in range(copies):
        ws.append((torch.from_numpy(w.w_packed.view(np.int32)).to(dev),
                   torch.from_numpy(w.scales.view(np.int16)).to(dev),
                   torch.from_numpy(w.biases.view(np.int16)).to(dev)))
    xt = torch.from_numpy(x.view(np.int16)).to(dev)
    yt = torch.empty((M, N), dtype=torch.int16, device=dev)
    kernel = {"auto": aq.AQ_KERNEL_AUTO, "qmv": aq.AQ_KERNEL_QMV, "qmm": aq.AQ_KERNEL_QMM}[args.kernel]
    stream = torch.cuda.current_stream(dev)

    xws = torch.empty(max(1, aq.aq_matmul_workspace_bytes(M, K)), dtype=torch.uint8, device=dev)

    def launch(i):
        wt, st, bt = ws[i % copies]
        if args.workspace:
            rc = lib.aq_matmul_bf16_ws(xt.data_ptr(), wt.data_ptr(), st.data_ptr(), bt.data_ptr(), yt.data_ptr(), M,
                                       N, K, 64, bits, xws.data_ptr(), xws.numel(), stream.cuda_stream)
        else:
            rc = lib.aq_matmul_bf16_ex(xt.data_ptr(), wt.data_ptr(), st.data_ptr(), bt.data_ptr(), yt.data_ptr(), M,
                                       N, K, 64, bits, kernel, 0, stream.cuda_stream)
        if rc != aq.AQ_OK:
            raise aq.AqError(rc, "matmul call")

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        launch(args.warmup + i)
    e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    hbm_peak, bf16_peak, _, _ = load_peaks()
    gbs = alg_bytes(M, N, K, bits) / (us * 1e-6) / 1e9
    tflops = 2.0 * M * N * K / (us * 1e-6) / 1e12
    print(json.dumps({"case": [M, N, K], "bits": bits, "kernel": args.kernel, "us_per_call": round(us, 3), "gbs": round(gbs, 1),
                      "hbm_frac": round(gbs / hbm_peak, 4), "tflops": round(tflops, 2),
                      "bf16_frac": round(tflops / bf16_peak, 4), "weight_copies": copies}), flush=True)


def run_case_other(args):
    """One NVFP4 shape (--nvfp4-case M,N,K) or one Mixtral-shaped MoE prefill
    matrix (--moe-case w1_gate|w3_up|w2_down: 2048 tokens, top-2 of 8 experts),
    timed through the C ABI with CUDA events; the ncu targets of those kernels."""
    import torch

    import affine_bit_quantized_gb300 as aq
    from affine_bit_quantized_gb300 import _build

    dev = torch.device("cuda", 0)
    _build.build_library()
    lib = aq.load()
    stream = torch.cuda.current_stream(dev)
    if args.nvfp4_case:
        M, N, K = (int(v) for v in args.nvfp4_case.split(","))
        w = synth.make_nvfp4_weights(N, K, 1)
        copies = max(1, min(64, -(-3 * 129 * 2**20 // (w.w_packed.nbytes + w.scales.nbytes))))
        ws = [(torch.from_numpy(w.w_packed.view(np.int32)).to(dev), torch.from_numpy(w.scales).to(dev))
              for _ in range(copies)]
        xt = torch.from_numpy(synth.make_x(M, K, 1).view(np.int16)).to(dev)
        yt = torch.empty((M, N), dtype=torch.int16, device=dev)

        def launch(i):
            wt, st = ws[i % copies]
            rc = lib.aq_matmul_nvfp4_bf16(xt.data_ptr(), wt.data_ptr(), st.data_ptr(), w.global_scale, yt.data_ptr(),
                                          M, N, K, 0, stream.cuda_stream)
            if rc != aq.AQ_OK:
                raise aq.AqError(rc, "aq_matmul_nvfp4_bf16")
        work = {"case": ["nvfp4", M, N, K], "bytes": alg_bytes(M, N, K)}
    else:
        name, N, K = [m for m in synth.MIXTRAL_EXPERT_MATS if m[0] == args.moe_case][0]
        T, E, top_k = 2048, synth.MIXTRAL_EXPERTS, synth.MIXTRAL_TOP_K
        lhs, rhs = synth.make_routing(T, E, top_k, synth.seed_for(6, 0, 9))
        ew = synth.ExpertWeights(E, N, K, synth.seed_for(6, 0, 0))
        wt = torch.from_numpy(ew.w_packed.view(np.int32)).to(dev)
        st = torch.from_numpy(ew.scales.view(np.int16)).to(dev)
        bt = torch.from_numpy(ew.biases.view(np.int16)).to(dev)
        xt = torch.from_numpy(synth.make_x(T, K, 1).view(np.int16)).to(dev)
        lt, rt = torch.from_numpy(lhs).to(dev), torch.from_numpy(rhs).to(dev)
        R = int(lhs.size)
        yt = torch.empty((R, N), dtype=torch.int16, device=dev)
        wsp = torch.empty(aq.aq_gather_qmm_workspace_bytes(R, K, E), dtype=torch.uint8, device=dev)

        def launch(i):
            rc = lib.aq_gather_qmm_bf16(xt.data_ptr(), wt.data_ptr(), st.data_ptr(), bt.data_ptr(), lt.data_ptr(),
                                        rt.data_ptr(), yt.data_ptr(), R, T, N, K, E, 64, 4, wsp.data_ptr(), wsp.numel(),
                                        stream.cuda_stream)
            if rc != aq.AQ_OK:
                raise aq.AqError(rc, "aq_gather_qmm_bf16")
        work = {"case": ["moe", name, T, E, top_k, N, K], "flops": 2.0 * R * N * K}
    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        launch(args.warmup + i)
    e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    out = {"case": work["case"], "us_per_call": round(us, 3)}
    if "bytes" in work:
        out["gbs"] = round(work["bytes"] / (us * 1e-6) / 1e9, 1)
    else:
        out["tflops"] = round(work["flops"] / (us * 1e-6) / 1e12, 1)
    print(json.dumps(out), flush=True)


def check_side_rates(per_matrix, small_batch, eight_bit, qmm, nvfp4, moe, read_peak, bf16_peak):
    """A side measurement far above its ceiling timed launches that did no work
    (a capture that recorded nothing, a call that returned early): refuse to
    print it.  Bandwidths are held against the measured read ceiling, tensor
    rates against the bf16 burst peak, each with 50 % to spare."""
    bad = []
    for sec in (per_matrix, small_batch, eight_bit, nvfp4):
        for name, e in (sec or {}).items():
            if "gbs" in e and e["gbs"] > 1.5 * read_peak:
                bad.append(f"{name}: {e['gbs']} GB/s")
    for sec in (qmm, moe):
        for name, e in (sec or {}).items():
            for key in ("tflops", "without_workspace_tflops"):
                if key in e and e[key] > 1.5 * bf16_peak:
                    bad.append(f"{name}: {e[key]} TFLOP/s")
    if bad:
        raise RuntimeError("side measurements above any ceiling (no work timed): " + "; ".join(bad))


def kernel_source_hash() -> str:
    """Hash of the chained kernel's sources with comments and blank space taken
    out (an edit of a comment leaves the captured traffic valid)."""
    h = hashlib.sha256()
    for name in ("qmv_chain.cu", "qmv_tma.cu", "qmv_consumer.cuh", "nvfp4_consumer.cuh", "aq_ptx.cuh"):
        with open(os.path.join(ROOT, "affine_bit_quantized_gb300", "csrc", name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def committed_traffic():
    """Per-step DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "qmv_chain_decode_step_dram_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_step"])
    except Exception:
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--layers", type=int, default=32, help="decoder layers in the step (32 = the workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step-only", action="store_true",
                    help="time the decode step (and its end-to-end form) only, without the side measurements")
    ap.add_argument("--case", default=None,
                    help="M,N,K: time one matrix shape instead of the decode step (also the ncu target)")
    ap.add_argument("--kernel", choices=("auto", "qmv", "qmm"), default="auto", help="kernel for --case")
    ap.add_argument("--bits", type=int, choices=(4, 8), default=4, help="code width for --case")
    ap.add_argument("--nvfp4-case", default=None, help="M,N,K: time one NVFP4 shape (an ncu target)")
    ap.add_argument("--moe-case", default=None, choices=[m[0] for m in synth.MIXTRAL_EXPERT_MATS],
                    help="time one MoE prefill matrix (2048 tokens, top-2 of 8 experts; an ncu target)")
    ap.add_argument("--workspace", action="store_true",
                    help="--case through aq_matmul_bf16_ws (x converted once for the tensor-core kernel)")
    ap.add_argument("--step-impl", choices=("chain", "graph"), default="chain",
                    help="decode step as one persistent chained launch (aq_chain_run) or as a CUDA graph of "
                         "one aq_matmul_bf16_ex launch per matrix; the other is reported as 'alt'")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local_rank = rank_env()

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if args.case:
        run_case(args)
        return
    if args.nvfp4_case or args.moe_case:
        run_case_other(args)
        return

    import torch
    import torch.distributed as dist

    import affine_bit_quantized_gb300 as aq
    from affine_bit_quantized_gb300 import _build

    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    _build.build_library()
    lib = aq.load()

    hbm_peak, bf16_peak, bf16_sus, peak_src = load_peaks()

    # ---- workload (generated on the host from the seeded recipe, uploaded once)
    cpu_layers = {0, 1} if (rank == 0 and world == 1 and not args.no_cpu_baseline and not args.step_only) else set()
    ds = DecodeStep(dev, args.layers, keep_host=bool(cpu_layers), host_layers=cpu_layers)
    mats, launches = ds.mats, ds.launches
    offs, _ = x_layout(args.layers)
    x_host, x_pinned, x_dev, y_dev, y_offs = ds.x_host, ds.x_pinned, ds.x, ds.y, ds.y_offsets
    weights = {(m[0], m[1]): ds.weights[i] for i, m in enumerate(mats)}
    host_keep = {(mats[i][0], mats[i][1]): w for i, w in ds.host_weights.items()}
    logits_pinned = torch.empty(mats[-1][3], dtype=torch.int16).pin_memory()
    step_bytes = sum(alg_bytes(1, N, K) for (_, _, _, N, K, _) in mats)
    enqueue = ds.enqueue
    # the step as a CUDA graph of one launch per matmul (k, v beside q and up
    # beside gate as parallel branches), reported as the alternative
    graph = ds.capture_graph()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    gpu_id = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    clocks = ClockSampler(gpu_id)

    # ---- the same step as one chained launch over the same buffers
    cur = torch.cuda.current_stream(dev)

    def chain_step():
        ds.run_chain(cur.cuda_stream)

    step_fns = {"chain": chain_step, "graph": graph.replay}
    step = step_fns[args.step_impl]
    alt_impl = "graph" if args.step_impl == "chain" else "chain"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def time_steps(fn, n):
        barrier()
        e0.record(cur)
        for _ in range(n):
            fn()
        e1.record(cur)
        e1.synchronize()
        return e0.elapsed_time(e1) / n

    # ---- device-resident timing (value)
    for _ in range(args.warmup):
        step()
    barrier()
    clocks.start()
    ms_step = time_steps(step, args.steps)
    clk = clocks.stop()
    barrier()
    ms_step = max_over_ranks(ms_step, world, dev)
    for _ in range(args.warmup):
        step_fns[alt_impl]()
    ms_alt = max_over_ranks(time_steps(step_fns[alt_impl], max(3, min(args.steps, 500))), world, dev)
    # the chain with every group's completion released (AQ_CHAIN_RELEASE on every matmul):
    # what the step costs when each matmul reads the previous group's output
    rel_plan, rel_ws = ds.released_plan()

    def chain_released():
        ds.run_chain(cur.cuda_stream, rel_plan)

    for _ in range(args.warmup):
        chain_released()
    ms_rel = max_over_ranks(time_steps(chain_released, max(3, min(args.steps, 500))), world, dev)
    del rel_ws
    if aq.aq_read_device_status(cur.cuda_stream) != aq.AQ_OK:
        raise RuntimeError("a bounded device-side wait expired during the timed steps")

    # ---- read-only streaming ceiling of this device: TMA bulk reads of a 4 GiB
    # buffer with no arithmetic (aq_read_probe), best of 5 runs of 10 launches
    probe_buf = torch.empty(4 << 30, dtype=torch.uint8, device=dev)

    def probe_once():
        rc = aq.aq_read_probe(probe_buf.data_ptr(), probe_buf.numel(), cur.cuda_stream)
        if rc != aq.AQ_OK:
            raise aq.AqError(rc, "aq_read_probe")

    for _ in range(3):
        probe_once()
    read_peak = max(probe_buf.numel() / (time_steps(probe_once, 10) * 1e-3) / 1e9 for _ in range(5))
    del probe_buf
    if aq.aq_read_device_status(cur.cuda_stream) != aq.AQ_OK:
        raise RuntimeError("a bounded device-side wait expired in the read probe")

    # ---- end to end: inputs copied in from pinned host memory, logits read back, every step
    h2d = x_pinned.numel() * 2
    d2h = logits_pinned.numel() * 2
    logits_dev = y_dev[y_offs[-1]:y_offs[-1] + mats[-1][3]]

    def e2e_step():
        x_dev.copy_(x_pinned, non_blocking=True)
        step()
        logits_pinned.copy_(logits_dev, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    ms_e2e = max_over_ranks(time_steps(e2e_step, args.steps), world, dev)

    def side_sections():
        """Per-matrix, small-batch, 8-bit, tensor-core, NVFP4 and MoE measurements beside the step."""
        def sh():
            """The stream the next launch goes to (the capture stream while a graph is captured)."""
            return torch.cuda.current_stream(dev).cuda_stream

        def graph_us(enqueue_all, n_calls, reps=5):
            """Device time per call of n_calls launches, captured once as a CUDA graph and
            replayed: launches with programmatic dependent launch, no host work in between (a
            Python loop of single calls is bound by the host at these sizes)."""
            for _ in range(2):
                enqueue_all()
            torch.cuda.synchronize(dev)
            cap = torch.cuda.Stream(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                enqueue_all()
            g.replay()
            torch.cuda.synchronize(dev)
            e0.record(cur)
            for _ in range(reps):
                g.replay()
            e1.record(cur)
            e1.synchronize()
            del g
            return e0.elapsed_time(e1) * 1e3 / (reps * n_calls)

        def time_calls(launch, n_calls, reps=5):
            def enqueue_all():
                for i in range(n_calls):
                    launch(i)
            return graph_us(enqueue_all, n_calls, reps)

        # ---- per-matrix kernel times (the 32 layer copies of each shape back to back)
        per_matrix = {}
        for j, (name, N, K) in enumerate(synth.LLAMA8B_LAYER + (synth.LLAMA8B_LM_HEAD,)):
            sel = {i for i, m in enumerate(mats) if (m[2] == name)}
            reps = 5 if len(sel) > 1 else 20
            us = graph_us(lambda sel=sel: enqueue(sh(), sel), len(sel), reps)
            per_matrix[name] = {"N": N, "K": K, "us_per_call": round(us, 3),
                                "gbs": round(alg_bytes(1, N, K) / (us * 1e-6) / 1e9, 1)}

        # ---- small batches (the multi-row decode path): M in {2, 4, 8, 16} over the layer shapes
        # and lm_head, on the step's copies (32 distinct weights per layer shape: no L2 reuse; the
        # one lm_head, 296 MB, is larger than L2)
        small_batch = {}
        for M in (2, 4, 8, 16):
            for j, (name, N, K) in enumerate(synth.LLAMA8B_LAYER + (synth.LLAMA8B_LM_HEAD,)):
                lm = name == "lm_head"
                xb = torch.from_numpy(synth.make_x(M, K, synth.seed_for(3, M, j)).view(np.int16)).to(dev)
                yb = torch.empty((M, N), dtype=torch.int16, device=dev)
                ws = [weights[(args.layers, 0)]] if lm else [weights[(layer, j)] for layer in range(args.layers)]

                def launch_sb(i, ws=ws, xb=xb, yb=yb, M=M, N=N, K=K):
                    wt, st_, bt = ws[i % len(ws)]
                    rc = lib.aq_matmul_bf16_ex(xb.data_ptr(), wt.data_ptr(), st_.data_ptr(), bt.data_ptr(), yb.data_ptr(),
                                               M, N, K, 64, 4, aq.AQ_KERNEL_AUTO, aq.AQ_FLAG_PDL, sh())
                    if rc != aq.AQ_OK:
                        raise aq.AqError(rc, "aq_matmul_bf16_ex")

                us = time_calls(launch_sb, 4 if lm else len(ws))
                small_batch[f"M{M}_{name}"] = {"M": M, "N": N, "K": K, "us_per_call": round(us, 3),
                                               "gbs": round(alg_bytes(M, N, K) / (us * 1e-6) / 1e9, 1)}

        def copies_for(nbytes):
            """Distinct device copies of a matrix whose cycle spans at least 3 x L2 (129 MB)."""
            return max(2, min(128, -(-3 * 129 * 2**20 // nbytes)))

        # ---- 8-bit codes (same shapes, M = 1): device copies of each weight matrix cycled over >= 3 x L2
        eight_bit = {}
        for j, (name, N, K) in enumerate(synth.LLAMA8B_LAYER + (synth.LLAMA8B_LM_HEAD,)):
            w8 = synth.make_weights(N, K, synth.seed_for(6, 0, j), bits=8)
            base = (torch.from_numpy(w8.w_packed.view(np.int32)).to(dev), torch.from_numpy(w8.scales.view(np.int16)).to(dev),
                    torch.from_numpy(w8.biases.view(np.int16)).to(dev))
            ws8 = [base] + [tuple(t.clone() for t in base) for _ in range(copies_for(N * K * 17 // 16) - 1)]
            x8 = torch.from_numpy(synth.make_x(1, K, synth.seed_for(6, 1, j)).view(np.int16)).to(dev)
            y8 = torch.empty((1, N), dtype=torch.int16, device=dev)

            def launch8(i, ws8=ws8, x8=x8, y8=y8, N=N, K=K):
                wt, st_, bt = ws8[i % len(ws8)]
                rc = lib.aq_matmul_bf16_ex(x8.data_ptr(), wt.data_ptr(), st_.data_ptr(), bt.data_ptr(), y8.data_ptr(),
                                           1, N, K, 64, 8, aq.AQ_KERNEL_AUTO, aq.AQ_FLAG_PDL, sh())
                if rc != aq.AQ_OK:
                    raise aq.AqError(rc, "aq_matmul_bf16_ex")

            us = time_calls(launch8, len(ws8))
            eight_bit[name] = {"N": N, "K": K, "us_per_call": round(us, 3),
                               "gbs": round(alg_bytes(1, N, K, 8) / (us * 1e-6) / 1e9, 1)}
            del ws8, base

        # ---- prefill-sized tensor-core GEMM (qmm): M in {256, 2048}, (K, N) in {(4096, 14336), (14336, 4096)},
        # 4-bit codes (the workload) and 8-bit codes
        qmm = {}
        for bits in (4, 8):
            for (K, N, label) in QMM_SHAPES:
                w = synth.make_weights(N, K, synth.seed_for(5, 0, 0 if N == 14336 else 1), bits=bits)
                copies = 4   # 4 x 33 MB (4-bit) of distinct weights > L2 between consecutive launches
                ws = [(torch.from_numpy(w.w_packed.view(np.int32)).to(dev), torch.from_numpy(w.scales.view(np.int16)).to(dev),
                       torch.from_numpy(w.biases.view(np.int16)).to(dev)) for _ in range(copies)]
                for M in QMM_M:
                    xq = torch.from_numpy(synth.make_x(M, K, synth.seed_for(5, M, 9)).view(np.int16)).to(dev)
                    yq = torch.empty((M, N), dtype=torch.int16, device=dev)

                    xws = torch.empty(aq.aq_matmul_workspace_bytes(M, K), dtype=torch.uint8, device=dev)

                    def qlaunch(i, ws=ws, xq=xq, yq=yq, M=M, N=N, K=K, bits=bits, xws=xws, use_ws=True):
                        wt, st, bt = ws[i % copies]
                        if use_ws:   # x converted once into the workspace (aq_matmul_bf16_ws)
                            rc = lib.aq_matmul_bf16_ws(xq.data_ptr(), wt.data_ptr(), st.data_ptr(), bt.data_ptr(),
                                                       yq.data_ptr(), M, N, K, 64, bits, xws.data_ptr(), xws.numel(),
                                                       cur.cuda_stream)
                        else:
                            rc = lib.aq_matmul_bf16_ex(xq.data_ptr(), wt.data_ptr(), st.data_ptr(), bt.data_ptr(),
                                                       yq.data_ptr(), M, N, K, 64, bits, aq.AQ_KERNEL_AUTO, 0,
                                                       cur.cuda_stream)
                        if rc != aq.AQ_OK:
                            raise aq.AqError(rc, "qmm call")

                    def time_q(use_ws, reps=10):
                        for i in range(3):
                            qlaunch(i, use_ws=use_ws)
                        torch.cuda.synchronize(dev)
                        e0.record(cur)
                        for i in range(reps):
                            qlaunch(i, use_ws=use_ws)
                        e1.record(cur)
                        e1.synchronize()
                        return e0.elapsed_time(e1) * 1e3 / reps

                    us = time_q(True)
                    us_plain = time_q(False)
                    tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
                    key = f"M{M}_K{K}_N{N}" + ("" if bits == 4 else "_8bit")
                    qmm[key] = {"us_per_call": round(us, 2), "tflops": round(tf, 1),
                                "frac_of_bf16_burst": round(tf / bf16_peak, 4),
                                "frac_of_bf16_sustained": round(tf / bf16_sus, 4),
                                "without_workspace_us": round(us_plain, 2),
                                "without_workspace_tflops": round(2.0 * M * N * K / (us_plain * 1e-6) / 1e12, 1)}
                    del xws
                del ws

        # ---- NVFP4 weights (E2M1 codes, E4M3 scale per 16, fp32 tensor scale), M = 1, the step's shapes:
        # device copies of each matrix cycled over >= 3 x L2 (0.5625 B per weight, as the affine 4-bit format)
        nvfp4 = {}
        for j, (name, N, K) in enumerate(synth.LLAMA8B_LAYER + (synth.LLAMA8B_LM_HEAD,)):
            wn = synth.make_nvfp4_weights(N, K, synth.seed_for(7, 0, j))
            base = (torch.from_numpy(wn.w_packed.view(np.int32)).to(dev), torch.from_numpy(wn.scales).to(dev))
            wsn = [base] + [tuple(t.clone() for t in base) for _ in range(copies_for(N * K * 9 // 16) - 1)]
            xn = torch.from_numpy(synth.make_x(1, K, synth.seed_for(7, 1, j)).view(np.int16)).to(dev)
            yn = torch.empty((1, N), dtype=torch.int16, device=dev)

            def launchn(i, wsn=wsn, xn=xn, yn=yn, N=N, K=K, g=wn.global_scale):
                wt, st_ = wsn[i % len(wsn)]
                rc = lib.aq_matmul_nvfp4_bf16(xn.data_ptr(), wt.data_ptr(), st_.data_ptr(), g, yn.data_ptr(), 1, N, K,
                                              aq.AQ_FLAG_PDL, sh())
                if rc != aq.AQ_OK:
                    raise aq.AqError(rc, "aq_matmul_nvfp4_bf16")

            us = time_calls(launchn, len(wsn))
            nvfp4[name] = {"N": N, "K": K, "us_per_call": round(us, 3),
                           "gbs": round(alg_bytes(1, N, K) / (us * 1e-6) / 1e9, 1)}
            del wsn, base

        # ---- the whole step with NVFP4 weights (same shapes, same 0.5625 bytes per weight, its
        # own seeds), as one chained launch like the headline step
        ds_nv = DecodeStep(dev, args.layers, fmt="nvfp4")

        def nv_step():
            ds_nv.run_chain(cur.cuda_stream)

        for _ in range(3):
            nv_step()
        ms_nv = time_steps(nv_step, max(3, min(args.steps, 20)))
        if aq.aq_read_device_status(cur.cuda_stream) != aq.AQ_OK:
            raise RuntimeError("a bounded device-side wait expired in the NVFP4 step")
        nvfp4["step_chain"] = {"layers": args.layers, "ms_per_step": round(ms_nv, 5),
                               "gbs": round(step_bytes / (ms_nv * 1e-3) / 1e9, 1),
                               "frac": round(step_bytes / (ms_nv * 1e-3) / 1e9 / hbm_peak, 4)}
        del ds_nv

        # ---- MoE prefill (expert-indexed matmul): Mixtral-8x7B-shaped experts, 2048 tokens routed
        # top-2 over 8 experts (4096 rows), one call = plan + row gather + tensor-core matmul
        moe = {}
        T_moe = 2048
        lhs, rhs = synth.make_routing(T_moe, synth.MIXTRAL_EXPERTS, synth.MIXTRAL_TOP_K, synth.seed_for(6, 0, 9))
        lt = torch.from_numpy(lhs).to(dev)
        rt = torch.from_numpy(rhs).to(dev)
        R_moe = int(lhs.size)
        for j, (name, N, K) in enumerate(synth.MIXTRAL_EXPERT_MATS):
            ew = synth.ExpertWeights(synth.MIXTRAL_EXPERTS, N, K, synth.seed_for(6, 0, 16 * j))
            wt = torch.from_numpy(ew.w_packed.view(np.int32)).to(dev)
            st = torch.from_numpy(ew.scales.view(np.int16)).to(dev)
            bt = torch.from_numpy(ew.biases.view(np.int16)).to(dev)
            xm = torch.from_numpy(synth.make_x(T_moe, K, synth.seed_for(6, 0, 8)).view(np.int16)).to(dev)
            ym = torch.empty((R_moe, N), dtype=torch.int16, device=dev)
            nws = aq.aq_gather_qmm_workspace_bytes(R_moe, K, synth.MIXTRAL_EXPERTS)
            wsm = torch.empty(nws, dtype=torch.uint8, device=dev)

            def mlaunch(i, wt=wt, st=st, bt=bt, xm=xm, ym=ym, wsm=wsm, N=N, K=K):
                rc = lib.aq_gather_qmm_bf16(xm.data_ptr(), wt.data_ptr(), st.data_ptr(), bt.data_ptr(), lt.data_ptr(),
                                            rt.data_ptr(), ym.data_ptr(), R_moe, T_moe, N, K, synth.MIXTRAL_EXPERTS, 64,
                                            4, wsm.data_ptr(), wsm.numel(), sh())
                if rc != aq.AQ_OK:
                    raise aq.AqError(rc, "aq_gather_qmm_bf16")

            us = time_calls(mlaunch, 4)
            tf = 2.0 * R_moe * N * K / (us * 1e-6) / 1e12
            moe[name] = {"tokens": T_moe, "experts": synth.MIXTRAL_EXPERTS, "top_k": synth.MIXTRAL_TOP_K, "rows": R_moe,
                         "N": N, "K": K, "us_per_call": round(us, 2), "tflops": round(tf, 1),
                         "frac_of_bf16_burst": round(tf / bf16_peak, 4)}
            del wt, st, bt, ew, wsm
        return per_matrix, small_batch, eight_bit, qmm, nvfp4, moe

    if args.step_only:
        per_matrix = small_batch = eight_bit = qmm = nvfp4 = moe = None
    else:
        per_matrix, small_batch, eight_bit, qmm, nvfp4, moe = side_sections()
        check_side_rates(per_matrix, small_batch, eight_bit, qmm, nvfp4, moe, read_peak, bf16_peak)

    # ---- CPU baseline: the oracle on two layers of the same workload, host cores
    cpu = None
    if cpu_layers:
        import oracle
        threads = oracle.default_threads()
        done_bytes, passes, t0 = 0, 0, time.perf_counter()
        # layers 0-1 of the step, repeated until at least 10 s of CPU work (at most 50 passes)
        while passes < 50 and (passes == 0 or time.perf_counter() - t0 < 10.0):
            for (layer, j), w in sorted(host_keep.items()):
                name = synth.LLAMA8B_LAYER[j][0]
                xo, K, xseed = offs[(layer, ROLE_OF[name])]
                x = x_host[xo:xo + K].reshape(1, K)
                oracle.matmul(x, w.w_packed, w.scales, w.biases, 1, w.N, w.K, nthreads=threads)
                done_bytes += alg_bytes(1, w.N, w.K)
            passes += 1
        dt = time.perf_counter() - t0
        cpu = {"value": round(done_bytes / dt / 1e9, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"layers 0-1 of the step ({len(host_keep)} matrices, "
                         f"{sum(w.N * w.K for w in host_keep.values()) / 1e6:.0f} M weights), M=1, fp64, "
                         f"{passes} passes",
               "seconds": round(dt, 2)}

    gbs = job_rate(world, step_bytes, ms_step * 1e-3) / 1e9
    gbs_e2e = job_rate(world, step_bytes, ms_e2e * 1e-3) / 1e9
    traffic = committed_traffic()
    line = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": args.layers, "M": 1, "bytes_per_step": step_bytes,
                   "matmuls_per_step": len(launches), "step_impl": args.step_impl,
                   "step_impl_desc": {"chain": "one cooperative persistent launch (aq_chain_run); a dependent "
                                               "matmul starts only after every tile of the previous dependency "
                                               "group is stored (completion counters); the activation rows live "
                                               "in their own buffer, so no group's completion needs a memory "
                                               "release (chain_released: with it)",
                                      "graph": "CUDA graph of one launch per matmul (k, v beside q and up beside "
                                               "gate as parallel branches), programmatic dependent launch"
                                      }[args.step_impl],
                   "l2": "inputs larger than L2 (4.22 GB of weights per step vs 129 MB L2)",
                   "parallelism": f"replicas x{world}"},
        "tok_s": round(world * 1e3 / ms_step, 1),
        "pct_of_hbm_peak": round(100 * gbs / world / hbm_peak, 1),
        "roofline": {"bound": "hbm", "achieved": round(step_bytes / (ms_step * 1e-3) / 1e9, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(step_bytes / (ms_step * 1e-3) / 1e9 / hbm_peak, 4),
                     "traffic": traffic if args.step_impl == "chain" else None,
                     "kernel": {"chain": "qmv_chain_kernel (the one launch of the step)",
                                "graph": "qmv_tma_kernel (every launch of the step)"}[args.step_impl],
                     "peak_source": f"{peak_src} hbm_gbs (copy)",
                     "peak_read": round(read_peak, 1),
                     "frac_read": round(step_bytes / (ms_step * 1e-3) / 1e9 / read_peak, 4),
                     "peak_read_source": "aq_read_probe on this device: TMA bulk reads of a 4 GiB buffer, "
                                         "no arithmetic, best of 5 x 10 launches"},
        "e2e": {"value": round(gbs_e2e, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e, 5)},
        "gpu_launches": args.steps * (1 if args.step_impl == "chain" else len(launches)),
        "alt": {"step_impl": alt_impl, "ms_per_step": round(ms_alt, 5),
                "value": round(world * step_bytes / (ms_alt * 1e-3) / 1e9, 1)},
        "chain_released": {"ms_per_step": round(ms_rel, 5),
                           "value": round(world * step_bytes / (ms_rel * 1e-3) / 1e9, 1),
                           "groups_released": int(rel_plan.reserved[3]),
                           "desc": "the timed chain with AQ_CHAIN_RELEASE on every matmul: each dependency "
                                   "group's completion published with a GPU-scope release"},
        "clocks": clk,
        "per_matrix": per_matrix,
        "small_batch": small_batch,
        "eight_bit": eight_bit,
        "nvfp4": nvfp4,
        "moe_prefill": moe,
        "qmm": qmm,
    }
    for k in ("per_matrix", "small_batch", "eight_bit", "nvfp4", "moe_prefill", "qmm"):
        if line[k] is None:
            del line[k]
    if cpu:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
