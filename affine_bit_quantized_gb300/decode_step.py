"""The Llama-3.1-8B-shaped decode step as a workload: which matmuls, in which
order, from which seeds, reading which activation row and writing where.

A step is every weight matrix of ``layers`` decoder layers (q, k, v, o, gate,
up, down; 4-bit codes, group 64, each layer drawn from its own seeds) plus
lm_head, each multiplied by one bf16 activation row (M = 1).  k and v read q's
input and up reads gate's, so in a chain they are flagged independent of the
matmul before them; every other matmul waits for the one before it.

This module lays the step out and marshals it onto the device for the chained
kernel (``aq_chain_prepare`` / ``aq_chain_run``) and for one launch per matmul
(``aq_matmul_bf16_ex``).  It holds none of the method's arithmetic: the inputs
come from ``synth``, the products from the library.  The benchmark times this
step and the tests compare its outputs with the oracle, so both see the same
launch.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import _lib as aq
from . import synth

CONFIG_ID = 4          # workload number of the full decode step in the seed rule
N_ROLES = 4            # activations per layer: attention in, attention out, MLP in, MLP activation
ROLE_OF = {"q_proj": 0, "k_proj": 0, "v_proj": 0, "o_proj": 1, "gate_proj": 2, "up_proj": 2, "down_proj": 3}
ROLE_K = (4096, 4096, 4096, 14336)
INDEPENDENT = ("k_proj", "v_proj", "up_proj")


def step_matrices(layers: int):
    """(layer, j, name, N, K, seed) of every matrix of the step, in chain order."""
    out = []
    for layer in range(layers):
        for j, (name, N, K) in enumerate(synth.LLAMA8B_LAYER):
            out.append((layer, j, name, N, K, synth.seed_for(CONFIG_ID, layer, j)))
    name, N, K = synth.LLAMA8B_LM_HEAD
    out.append((layers, 0, name, N, K, synth.seed_for(CONFIG_ID, layers, 0)))
    return out


def x_layout(layers: int):
    """{(layer, role): (offset in elements, K, seed)} of every activation row
    inside one contiguous x buffer, and the buffer's length.  lm_head's input is
    role 0 of layer ``layers``."""
    offs, pos = {}, 0
    for layer in range(layers):
        for role, K in enumerate(ROLE_K):
            offs[(layer, role)] = (pos, K, synth.seed_for(CONFIG_ID, layer, 8 + role))
            pos += K
    offs[(layers, 0)] = (pos, synth.LLAMA8B_LM_HEAD[2], synth.seed_for(CONFIG_ID, layers, 8))
    pos += synth.LLAMA8B_LM_HEAD[2]
    return offs, pos


def x_offset(layers: int, mat) -> int:
    """Element offset of the activation row matrix ``mat`` (a step_matrices entry) reads."""
    offs, _ = x_layout(layers)
    layer, _, name = mat[0], mat[1], mat[2]
    return offs[(layer, 0 if name == "lm_head" else ROLE_OF[name])][0]


def independent_flags(mats):
    return [m[2] in INDEPENDENT for m in mats]


def host_x(layers: int) -> np.ndarray:
    """Every activation row of the step, as uint16 bf16 bit patterns, in x_layout order."""
    offs, n = x_layout(layers)
    x = np.empty(n, np.uint16)
    for (pos, K, seed) in offs.values():
        x[pos:pos + K] = synth.make_x(1, K, seed)[0]
    return x


class DecodeStep:
    """The step's buffers on one CUDA device: every weight matrix (its own
    allocation), all activation rows in one buffer ``x``, all outputs in one
    buffer ``y`` (matmul i at ``y_offsets[i]``), the chain descriptors and a
    prepared chain plan.

    keep_host: keep the host copies of the weights (``host_weights[i]``, for a
    comparison with the oracle); ``host_layers`` limits that to some layers.

    fmt: "affine4" (4-bit codes, groups of 64, bf16 scales and biases) or
    "nvfp4" (E2M1 codes, E4M3 scales per 16 codes, one fp32 scale per matrix:
    the same 0.5625 bytes per weight); a weight tuple is then (codes, E4M3
    scales, the fp32 scale as a one-element device tensor).
    """

    def __init__(self, device, layers: int = synth.LLAMA8B_LAYERS, keep_host: bool = False, host_layers=None,
                 threads: int | None = None, fmt: str = "affine4"):
        import torch

        if fmt not in ("affine4", "nvfp4"):
            raise ValueError(f"unknown weight format {fmt!r}")
        self.fmt = fmt
        self.device = device
        self.layers = layers
        self.mats = step_matrices(layers)
        self.independent = independent_flags(self.mats)
        self.x_host = host_x(layers)
        self.x_pinned = torch.from_numpy(self.x_host.view(np.int16)).pin_memory()
        self.x = self.x_pinned.to(device)
        self.y_offsets, pos = [], 0
        for m in self.mats:
            self.y_offsets.append(pos)
            pos += m[3]
        self.y = torch.empty(pos, dtype=torch.int16, device=device)
        self.host_weights = {}
        self.weights = [None] * len(self.mats)
        pool = ThreadPoolExecutor(threads or max(1, min(16, os.cpu_count() or 1)))

        def gen(i):
            _, _, _, N, K, seed = self.mats[i]
            if fmt == "nvfp4":
                return i, synth.make_nvfp4_weights(N, K, seed)
            return i, synth.make_weights(N, K, seed)

        self.global_scales = [1.0] * len(self.mats)
        for i, w in pool.map(gen, range(len(self.mats))):
            if fmt == "nvfp4":
                self.global_scales[i] = float(w.global_scale)
                self.weights[i] = (torch.from_numpy(w.w_packed.view(np.int32)).to(device),
                                   torch.from_numpy(w.scales).to(device),
                                   torch.tensor([w.global_scale], dtype=torch.float32, device=device))
            else:
                self.weights[i] = (torch.from_numpy(w.w_packed.view(np.int32)).to(device),
                                   torch.from_numpy(w.scales.view(np.int16)).to(device),
                                   torch.from_numpy(w.biases.view(np.int16)).to(device))
            if keep_host and (host_layers is None or self.mats[i][0] in host_layers):
                self.host_weights[i] = w
        pool.shutdown()
        self.launches = []
        for i, m in enumerate(self.mats):
            _, _, _, N, K, _ = m
            wt, st, bt = self.weights[i]
            self.launches.append((self.x.data_ptr() + 2 * x_offset(layers, m), wt.data_ptr(), st.data_ptr(),
                                  bt.data_ptr(), self.y.data_ptr() + 2 * self.y_offsets[i], 1, N, K))
        self.descs = (aq.MatmulDesc * len(self.launches))(*[
            aq.MatmulDesc(xp, wp, sp, bp, yp, M, N, K, aq.AQ_CHAIN_INDEPENDENT if ind else 0)
            for (xp, wp, sp, bp, yp, M, N, K), ind in zip(self.launches, self.independent)])
        nbytes = aq.aq_chain_workspace_bytes(len(self.launches))
        self.chain_workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.plan = aq.ChainPlan()
        st = aq.aq_chain_prepare(self.descs, len(self.launches), 16 if fmt == "nvfp4" else 64, 4,
                                 self.chain_workspace.data_ptr(), nbytes, self.plan)
        if st != aq.AQ_OK:
            raise aq.AqError(st, "aq_chain_prepare")

    @property
    def count(self) -> int:
        return len(self.mats)

    def output(self, i: int):
        """Device view of matmul i's output row (int16 bit patterns of bf16)."""
        return self.y[self.y_offsets[i]:self.y_offsets[i] + self.mats[i][3]]

    def host_x_row(self, i: int) -> np.ndarray:
        """Matmul i's activation row, [1, K] uint16."""
        off = x_offset(self.layers, self.mats[i])
        return self.x_host[off:off + self.mats[i][4]].reshape(1, -1)

    def run_chain(self, stream_handle, plan=None) -> None:
        """The whole step as one persistent launch (aq_chain_run), on this
        step's plan or on ``plan`` (from ``released_plan``)."""
        st = aq.aq_chain_run(self.plan if plan is None else plan, stream_handle)
        if st != aq.AQ_OK:
            raise aq.AqError(st, "aq_chain_run")

    def released_plan(self):
        """(plan, workspace) of the same chain with AQ_CHAIN_RELEASE on every
        matmul: every dependency group's completion published with a GPU-scope
        release, as if each matmul read the previous group's output."""
        import torch

        descs = (aq.MatmulDesc * self.count)(*[
            aq.MatmulDesc(d.x, d.w_packed, d.scales, d.biases, d.y, d.M, d.N, d.K, d.flags | aq.AQ_CHAIN_RELEASE)
            for d in self.descs])
        nbytes = aq.aq_chain_workspace_bytes(self.count)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        plan = aq.ChainPlan()
        st = aq.aq_chain_prepare(descs, self.count, 16 if self.fmt == "nvfp4" else 64, 4, workspace.data_ptr(),
                                 nbytes, plan)
        if st != aq.AQ_OK:
            raise aq.AqError(st, "aq_chain_prepare")
        return plan, workspace

    def enqueue(self, stream_handle, sel=None, flags: int = aq.AQ_FLAG_PDL) -> None:
        """One launch per matmul (those in ``sel``, or all), in order:
        aq_matmul_bf16_ex, or aq_matmul_nvfp4_bf16 for NVFP4 weights."""
        lib = aq.load()
        for i, (xp, wp, sp, bp, yp, M, N, K) in enumerate(self.launches):
            if sel is not None and i not in sel:
                continue
            if self.fmt == "nvfp4":
                st = lib.aq_matmul_nvfp4_bf16(xp, wp, sp, self.global_scales[i], yp, M, N, K, flags, stream_handle)
            else:
                st = lib.aq_matmul_bf16_ex(xp, wp, sp, bp, yp, M, N, K, 64, 4, aq.AQ_KERNEL_AUTO, flags,
                                           stream_handle)
            if st != aq.AQ_OK:
                raise aq.AqError(st, "matmul launch")

    def capture_graph(self):
        """The step as a CUDA graph of one launch per matmul: k and v run as
        branches beside q (same input, no mutual dependency), up beside gate;
        along each branch, launches chain with programmatic dependent launch."""
        import torch

        dev = self.device
        cap_stream = torch.cuda.Stream(dev)
        side = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

        def enqueue_dag():
            main = torch.cuda.current_stream(dev)
            i = 0
            while i < self.count:
                group = [i]
                while i + len(group) < self.count and self.independent[i + len(group)]:
                    group.append(i + len(group))
                if len(group) == 1:
                    self.enqueue(main.cuda_stream, {i})
                else:
                    fork = torch.cuda.Event()
                    fork.record(main)
                    joins = []
                    for b, idx in enumerate(group[1:]):
                        side[b].wait_event(fork)
                        self.enqueue(side[b].cuda_stream, {idx})
                        ev = torch.cuda.Event()
                        ev.record(side[b])
                        joins.append(ev)
                    self.enqueue(main.cuda_stream, {group[0]})
                    for ev in joins:
                        main.wait_event(ev)
                i += len(group)

        with torch.cuda.stream(cap_stream):
            enqueue_dag()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap_stream):
            enqueue_dag()
        torch.cuda.synchronize(dev)
        return graph
