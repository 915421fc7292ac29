"""CPU oracle for the affine group-quantized matmul (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path never does: it shares no code,
header, table or helper with the oracle.

The arithmetic lives in ``aq_oracle.c`` (plain C, fp64, multithreaded); this
module compiles it with gcc on first use and wraps it with ctypes.  See the C
file's header for the definition it follows and the readings of the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "aq_oracle.c")
_SRCS = (_SRC, os.path.join(_HERE, "nvfp4_oracle.c"))
_LIB = os.path.join(_HERE, "liboracle_aq.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle_aq.so`` (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or any(os.path.getmtime(_LIB) < os.path.getmtime(s) for s in _SRCS):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
             "-std=c11", "-o", tmp, *_SRCS, "-lm", "-lpthread"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.aqo_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.aqo_bf16_to_double.restype = ctypes.c_double
            lib.aqo_double_to_bf16.argtypes = [ctypes.c_double]
            lib.aqo_double_to_bf16.restype = ctypes.c_uint16
            lib.aqo_double_to_bf16_array.argtypes = [P, I64, P]
            lib.aqo_double_to_bf16_array.restype = None
            lib.aqo_unpack.argtypes = [P, I64, I64, I, P]
            lib.aqo_pack.argtypes = [P, I64, I64, I, P]
            lib.aqo_dequant.argtypes = [P, P, P, I64, I64, I, I, P]
            lib.aqo_matmul.argtypes = [P, P, P, P, I64, I64, I64, I, I, P, P, I]
            lib.aqo_matmul_sampled.argtypes = [P, P, P, P, I64, I64, I64, I, I, P, P, I64, P, P, I]
            lib.aqo_quantize.argtypes = [P, I64, I64, I, I, P, P, P]
            D = ctypes.c_double
            F = ctypes.c_float
            lib.aqo_e2m1_to_double.argtypes = [ctypes.c_uint]
            lib.aqo_e2m1_to_double.restype = D
            lib.aqo_e4m3_to_double.argtypes = [ctypes.c_uint]
            lib.aqo_e4m3_to_double.restype = D
            lib.aqo_nvfp4_dequant.argtypes = [P, P, F, I64, I64, P]
            lib.aqo_nvfp4_matmul.argtypes = [P, P, P, F, I64, I64, I64, P, P]
            lib.aqo_nvfp4_matmul_sampled.argtypes = [P, P, P, F, I64, I64, I64, P, P, I64, P, P]
            lib.aqo_default_threads.argtypes = []
            for f in ("aqo_unpack", "aqo_pack", "aqo_dequant", "aqo_matmul", "aqo_matmul_sampled",
                      "aqo_quantize", "aqo_default_threads"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def default_threads() -> int:
    return int(_load().aqo_default_threads())


def bf16_to_double(h) -> np.ndarray:
    h = _c(h, np.uint16)
    lib = _load()
    return np.array([lib.aqo_bf16_to_double(int(v)) for v in h.ravel()]).reshape(h.shape)


def double_to_bf16(v) -> np.ndarray:
    """Round doubles to bf16 (nearest, ties to even) directly from double."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().aqo_double_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def unpack(w_packed, N: int, K: int, bits: int = 4) -> np.ndarray:
    w_packed = _c(w_packed, np.uint32)
    codes = np.empty((N, K), np.uint8)
    if _load().aqo_unpack(_ptr(w_packed), N, K, bits, _ptr(codes)):
        raise ValueError("unsupported bits")
    return codes


def pack(codes, bits: int = 4) -> np.ndarray:
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    out = np.empty((N, K * bits // 32), np.uint32)
    if _load().aqo_pack(_ptr(codes), N, K, bits, _ptr(out)):
        raise ValueError("unsupported bits")
    return out


def dequant(w_packed, scales, biases, N: int, K: int, group_size: int = 64, bits: int = 4) -> np.ndarray:
    w_packed, scales, biases = _c(w_packed, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    out = np.empty((N, K), np.float64)
    if _load().aqo_dequant(_ptr(w_packed), _ptr(scales), _ptr(biases), N, K, group_size, bits, _ptr(out)):
        raise ValueError("bad arguments")
    return out


def matmul(x, w_packed, scales, biases, M: int, N: int, K: int, group_size: int = 64, bits: int = 4,
           nthreads: int = 0):
    """Return (y_exact float64[M,N], y_bf16 uint16[M,N])."""
    x = _c(x, np.uint16)
    w_packed, scales, biases = _c(w_packed, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    y_exact = np.empty((M, N), np.float64)
    y_bf16 = np.empty((M, N), np.uint16)
    rc = _load().aqo_matmul(_ptr(x), _ptr(w_packed), _ptr(scales), _ptr(biases), M, N, K, group_size,
                            bits, _ptr(y_exact), _ptr(y_bf16), nthreads)
    if rc:
        raise ValueError(f"oracle matmul failed ({rc})")
    return y_exact, y_bf16


def matmul_sampled(x, w_packed, scales, biases, M: int, N: int, K: int, idx_m, idx_n,
                   group_size: int = 64, bits: int = 4, nthreads: int = 0):
    """The definition evaluated at the (idx_m[i], idx_n[i]) pairs only."""
    x = _c(x, np.uint16)
    w_packed, scales, biases = _c(w_packed, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    idx_m, idx_n = _c(idx_m, np.int64), _c(idx_n, np.int64)
    count = idx_m.size
    y_exact = np.empty(count, np.float64)
    y_bf16 = np.empty(count, np.uint16)
    rc = _load().aqo_matmul_sampled(_ptr(x), _ptr(w_packed), _ptr(scales), _ptr(biases), M, N, K,
                                    group_size, bits, _ptr(idx_m), _ptr(idx_n), count, _ptr(y_exact),
                                    _ptr(y_bf16), nthreads)
    if rc:
        raise ValueError(f"oracle sampled matmul failed ({rc})")
    return y_exact, y_bf16


def gather_matmul(x, w_packed, scales, biases, lhs_indices, rhs_indices, N: int, K: int,
                  group_size: int = 64, bits: int = 4, nthreads: int = 0):
    """Expert-indexed matmul (MLX gather_qmm with the weights transposed, as in
    the MoE prefill path of "epic: CUDA (MLX backend) prefill and decode
    acceleration program", Diagnosis table and Phase 3): output row r is token
    row x[lhs_indices[r]] times dequant(W[rhs_indices[r]])^T.

    x uint16[T, K]; w_packed uint32[E, N, K*bits/32]; scales, biases
    uint16[E, N, K/group_size].  Written out plainly: the rows that share an
    expert are gathered and multiplied by that expert with ``matmul`` (the
    pinned definition), then scattered back to their row positions.
    Returns (y_exact float64[R, N], y_bf16 uint16[R, N])."""
    x = _c(x, np.uint16)
    lhs = np.asarray(lhs_indices, dtype=np.int64)
    rhs = np.asarray(rhs_indices, dtype=np.int64)
    R = lhs.size
    y_exact = np.zeros((R, N), np.float64)
    y_bf16 = np.zeros((R, N), np.uint16)
    for e in np.unique(rhs):
        rows = np.nonzero(rhs == e)[0]
        xe = x[lhs[rows]]
        ye, yb = matmul(xe, w_packed[e], scales[e], biases[e], rows.size, N, K, group_size, bits, nthreads)
        y_exact[rows] = ye
        y_bf16[rows] = yb
    return y_exact, y_bf16


def gather_matmul_sampled(x, w_packed, scales, biases, lhs_indices, rhs_indices, N: int, K: int, idx_r, idx_n,
                          group_size: int = 64, bits: int = 4, nthreads: int = 0):
    """``gather_matmul`` evaluated at the (idx_r[i], idx_n[i]) pairs only (for
    full-size checks): each sampled row is its token times its expert, through
    ``matmul_sampled``.  Returns (y_exact float64[S], y_bf16 uint16[S])."""
    x = _c(x, np.uint16)
    lhs = np.asarray(lhs_indices, dtype=np.int64)
    rhs = np.asarray(rhs_indices, dtype=np.int64)
    idx_r = np.asarray(idx_r, dtype=np.int64)
    idx_n = np.asarray(idx_n, dtype=np.int64)
    y_exact = np.zeros(idx_r.size, np.float64)
    y_bf16 = np.zeros(idx_r.size, np.uint16)
    for e in np.unique(rhs[idx_r]):
        sel = np.nonzero(rhs[idx_r] == e)[0]
        xe = x[lhs[idx_r[sel]]]                        # one x row per sample
        ye, yb = matmul_sampled(xe, w_packed[e], scales[e], biases[e], sel.size, N, K,
                                np.arange(sel.size), idx_n[sel], group_size, bits, nthreads)
        y_exact[sel] = ye
        y_bf16[sel] = yb
    return y_exact, y_bf16


# ---------------------------------------------------------------- NVFP4 (nvfp4_oracle.c)

def e2m1_to_double(code: int) -> float:
    """Value of one FP4 E2M1 code (0..15)."""
    return _load().aqo_e2m1_to_double(int(code))


def e4m3_to_double(byte: int) -> float:
    """Value of one FP8 E4M3 byte (NaN for S.1111.111)."""
    return _load().aqo_e4m3_to_double(int(byte))


def nvfp4_dequant(w_packed, scales, global_scale: float, N: int, K: int) -> np.ndarray:
    """w[n,k] = global * e4m3(scales[n, k/16]) * e2m1(q[n,k]) as float64[N, K]."""
    w_packed, scales = _c(w_packed, np.uint32), _c(scales, np.uint8)
    out = np.empty((N, K), np.float64)
    if _load().aqo_nvfp4_dequant(_ptr(w_packed), _ptr(scales), float(global_scale), N, K, _ptr(out)):
        raise ValueError("oracle nvfp4 dequant failed")
    return out


def nvfp4_matmul(x, w_packed, scales, global_scale: float, M: int, N: int, K: int):
    """y = x . w^T for NVFP4 weights (group 16, e4m3 scales, fp32 tensor scale).
    Returns (y_exact float64[M,N], y_bf16 uint16[M,N])."""
    x = _c(x, np.uint16)
    w_packed, scales = _c(w_packed, np.uint32), _c(scales, np.uint8)
    y_exact = np.empty((M, N), np.float64)
    y_bf16 = np.empty((M, N), np.uint16)
    if _load().aqo_nvfp4_matmul(_ptr(x), _ptr(w_packed), _ptr(scales), float(global_scale), M, N, K,
                                _ptr(y_exact), _ptr(y_bf16)):
        raise ValueError("oracle nvfp4 matmul failed")
    return y_exact, y_bf16


def nvfp4_matmul_sampled(x, w_packed, scales, global_scale: float, M: int, N: int, K: int, idx_m, idx_n):
    """``nvfp4_matmul`` at the (idx_m[i], idx_n[i]) pairs only."""
    x = _c(x, np.uint16)
    w_packed, scales = _c(w_packed, np.uint32), _c(scales, np.uint8)
    idx_m, idx_n = _c(idx_m, np.int64), _c(idx_n, np.int64)
    y_exact = np.empty(idx_m.size, np.float64)
    y_bf16 = np.empty(idx_m.size, np.uint16)
    if _load().aqo_nvfp4_matmul_sampled(_ptr(x), _ptr(w_packed), _ptr(scales), float(global_scale), M, N, K,
                                        _ptr(idx_m), _ptr(idx_n), idx_m.size, _ptr(y_exact), _ptr(y_bf16)):
        raise ValueError("oracle nvfp4 sampled matmul failed")
    return y_exact, y_bf16


def quantize(w, group_size: int = 64, bits: int = 4):
    """Min-max affine quantization; returns (w_packed, scales_bf16, biases_bf16)."""
    w = _c(w, np.float32)
    N, K = w.shape
    G = K // group_size
    wp = np.empty((N, K * bits // 32), np.uint32)
    s = np.empty((N, G), np.uint16)
    b = np.empty((N, G), np.uint16)
    if _load().aqo_quantize(_ptr(w), N, K, group_size, bits, _ptr(wp), _ptr(s), _ptr(b)):
        raise ValueError("bad arguments")
    return wp, s, b
