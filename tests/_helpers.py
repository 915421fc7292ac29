"""Shared test helpers: the pass criterion and host<->device marshalling."""
import numpy as np


def bf16_to_f64(h) -> np.ndarray:
    h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(v) -> np.ndarray:
    """Spacing of bf16 values at |v|: 2^(floor(log2|v|) - 7), and 2^-133 in the
    subnormal range (also used for v == 0)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126.0), -126.0)
    return np.exp2(e - 7.0)


def tolerance(y_ref_bits, rms=None) -> np.ndarray:
    """Per-element bound |y_gpu - y_ref| <= ulp_bf16(y_ref) + 1e-3 * RMS(y_ref),
    y_ref = the oracle's result rounded to bf16; RMS over the whole output (or
    the given estimate, for sampled outputs)."""
    r = bf16_to_f64(y_ref_bits)
    if rms is None:
        rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    return ulp_bf16(r) + 1e-3 * rms


def assert_parity(y_gpu_bits, y_ref_bits, rms=None, what=""):
    g = bf16_to_f64(y_gpu_bits)
    r = bf16_to_f64(y_ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    tol = tolerance(y_ref_bits, rms)
    err = np.abs(g - r)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst err/tol "
            f"{float(np.nanmax(err / tol)):.3g}; first {idx.tolist()} gpu {g[bad][:5]} ref {r[bad][:5]}")
    return float(np.max(err / tol)) if err.size else 0.0


# ---------------------------------------------------------------- torch marshalling

def to_dev_bf16(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(dev).view(torch.bfloat16)


def to_dev_u32(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).to(dev)


def from_dev_bf16(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def upload(x, w, dev):
    return (to_dev_bf16(x, dev), to_dev_u32(w.w_packed, dev), to_dev_bf16(w.scales, dev),
            to_dev_bf16(w.biases, dev))
