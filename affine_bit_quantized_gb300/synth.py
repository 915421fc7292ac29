"""Seeded synthetic inputs for the affine group-quantized matmul.

This module only draws random inputs; it holds none of the method's arithmetic
(no unpacking, no dequantization, no dot products).  Both the CUDA path and the
CPU oracle consume what it returns, so the two sides always see identical bytes.

Recipe (one case = one weight matrix W[N,K] plus an activation x[M,K]):

* packed codes: ``N * K * bits / 32`` uint32 words, each word uniform over
  [0, 2^32).  For 4-bit codes this is exactly "every code uniform in [0, 15]"
  (eight independent nibbles per word); for 8-bit codes, every code uniform in
  [0, 255].
* scales: bf16(U(0.004, 0.02) * 15 / (2^bits - 1)), one per group of ``group_size``
  along K (the 4-bit range; 8-bit codes cover the same weight range in finer steps).
* biases: bf16(-(2^bits - 1)/2 * scale + N(0, 0.002)), with ``scale`` the bf16 value, so
  that the dequantized weights are centred near zero.
* x: bf16(N(0, 1)).

bf16 values are returned as their uint16 bit patterns.  The bf16 rounding here
is round-to-nearest-even from float32 (numpy rounds float64 -> float32 first);
this double rounding only shapes the input distribution, never a result.

Random streams: ``numpy.random.Philox`` keyed through
``SeedSequence([seed, stream])``; stream 0 draws the weights (codes, then
scales, then bias noise), stream 1 draws x, stream 2 draws the MoE routing.
The seed of matrix j of layer l of workload c is ``1000*c + 16*l + j``; the tiny
correctness case uses seed 0.

MoE (expert-indexed) cases: E expert matrices of one shape stacked (expert e
from seed + e), T tokens of x, and a synthetic top-k routing: each token picks
k distinct experts uniformly at random; the rows (token, expert) are sorted by
expert, as a grouped prefill kernel consumes them.
"""
from __future__ import annotations

import dataclasses

import numpy as np

STREAM_WEIGHTS = 0
STREAM_X = 1
STREAM_ROUTING = 2


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(seed), int(stream)])))


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bit patterns."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(h) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
    return (h.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class QuantWeights:
    """A packed weight matrix: ``w_packed`` uint32[N, K*bits/32], ``scales``/``biases``
    bf16 bit patterns uint16[N, K/group_size]."""

    w_packed: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    N: int
    K: int
    group_size: int
    bits: int

    @property
    def nbytes(self) -> int:
        return self.w_packed.nbytes + self.scales.nbytes + self.biases.nbytes


def make_weights(N: int, K: int, seed: int, group_size: int = 64, bits: int = 4) -> QuantWeights:
    """Draw a packed weight matrix W[N,K] with the recipe in the module docstring."""
    if K % group_size or (K * bits) % 32:
        raise ValueError("K must be a multiple of group_size and of 32/bits")
    rng = _rng(seed, STREAM_WEIGHTS)
    words = K * bits // 32
    w_packed = rng.integers(0, 1 << 32, size=(N, words), dtype=np.uint32)
    G = K // group_size
    top = (1 << bits) - 1          # 15 for 4-bit codes, 255 for 8-bit
    s = f32_to_bf16_bits(rng.uniform(0.004, 0.02, size=(N, G)) * (15.0 / top))
    noise = rng.normal(0.0, 0.002, size=(N, G))
    b = f32_to_bf16_bits(-(top / 2.0) * bf16_bits_to_f32(s).astype(np.float64) + noise)
    return QuantWeights(w_packed, s, b, N, K, group_size, bits)


def make_x(M: int, K: int, seed: int) -> np.ndarray:
    """Draw activations x[M,K] = bf16(N(0,1)) as uint16 bit patterns."""
    rng = _rng(seed, STREAM_X)
    return f32_to_bf16_bits(rng.standard_normal((M, K)))


def seed_for(config: int, layer: int = 0, matrix: int = 0) -> int:
    """Seed of matrix ``matrix`` of layer ``layer`` in workload ``config`` (1-based)."""
    if config == 1:
        return 0
    return 1000 * config + 16 * layer + matrix


class ExpertWeights:
    """E packed weight matrices stacked: ``w_packed`` uint32[E, N, K*bits/32],
    ``scales``/``biases`` uint16[E, N, K/group_size] (expert e drawn with
    ``make_weights(N, K, seed + e)``)."""

    def __init__(self, E: int, N: int, K: int, seed: int, group_size: int = 64, bits: int = 4):
        ws = [make_weights(N, K, seed + e, group_size, bits) for e in range(E)]
        self.w_packed = np.stack([w.w_packed for w in ws])
        self.scales = np.stack([w.scales for w in ws])
        self.biases = np.stack([w.biases for w in ws])
        self.E, self.N, self.K, self.group_size, self.bits = E, N, K, group_size, bits


@dataclasses.dataclass
class NVFP4Weights:
    """NVFP4 weights: ``w_packed`` uint32[N, K/8] of FP4 E2M1 codes (lowest nibble
    = lowest k), ``scales`` uint8[N, K/16] of FP8 E4M3 block scales, and one fp32
    ``global_scale``."""

    w_packed: np.ndarray
    scales: np.ndarray
    global_scale: float
    N: int
    K: int


def make_nvfp4_weights(N: int, K: int, seed: int) -> NVFP4Weights:
    """Synthetic NVFP4 weights: every E2M1 code uniform over its 16 encodings,
    block scales uniform over the E4M3 encodings 0x48..0x7E (4 to 448, all
    finite and normal), global scale 2^-13 (weights of magnitude ~0.01-0.3)."""
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    rng = _rng(seed, STREAM_WEIGHTS)
    w_packed = rng.integers(0, 1 << 32, size=(N, K // 8), dtype=np.uint32)
    scales = rng.integers(0x48, 0x7F, size=(N, K // 16), dtype=np.uint8)
    return NVFP4Weights(w_packed, scales, 2.0 ** -13, N, K)


def make_routing(T: int, E: int, top_k: int, seed: int):
    """Synthetic top-k routing of T tokens over E experts: every token picks
    top_k distinct experts uniformly at random.  Returns int32 arrays
    (lhs, rhs) of T*top_k rows sorted by expert (stable, so by token within an
    expert): row r multiplies token lhs[r] by expert rhs[r]."""
    rng = _rng(seed, STREAM_ROUTING)
    picks = np.argsort(rng.random((T, E)), axis=1)[:, :top_k]      # top_k distinct experts per token
    tok = np.repeat(np.arange(T, dtype=np.int64), top_k)
    exp = picks.reshape(-1).astype(np.int64)
    order = np.lexsort((tok, exp))
    return tok[order].astype(np.int32), exp[order].astype(np.int32)


# Mixtral-8x7B-shaped MoE feed-forward (the pages' MoE prefill case): 8 experts,
# top-2 routing, (name, N, K) of each expert's matrices.
MIXTRAL_EXPERTS = 8
MIXTRAL_TOP_K = 2
MIXTRAL_EXPERT_MATS = (
    ("w1_gate", 14336, 4096),
    ("w3_up", 14336, 4096),
    ("w2_down", 4096, 14336),
)

# Llama-3.1-8B-shaped decode layer, (name, N, K): q, k, v, o, gate, up, down.
LLAMA8B_LAYER = (
    ("q_proj", 4096, 4096),
    ("k_proj", 1024, 4096),
    ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096),
    ("gate_proj", 14336, 4096),
    ("up_proj", 14336, 4096),
    ("down_proj", 4096, 14336),
)
LLAMA8B_LM_HEAD = ("lm_head", 128256, 4096)
LLAMA8B_LAYERS = 32
