"""ctypes binding of libaq.so: the same names as the C ABI, argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; there is no
Python or CPU fallback.  If the library has not been built this module raises
on first use.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from ._build import INCLUDE, LIB

AQ_OK = 0
AQ_ERR_INVALID_ARG = 1
AQ_ERR_UNSUPPORTED = 2
AQ_ERR_ALIGNMENT = 3
AQ_ERR_CUDA = 4
AQ_ERR_TIMEOUT = 5
AQ_ERR_BAD_INDEX = 6

AQ_KERNEL_AUTO = 0
AQ_KERNEL_QMV = 1
AQ_KERNEL_QMM = 2

AQ_FLAG_PDL = 1
AQ_FLAG_DEBUG_SKIP_COPY = 1 << 31
AQ_CHAIN_INDEPENDENT = 1
AQ_CHAIN_RELEASE = 2
AQ_CHAIN_DEBUG_SKIP_COPY = 0x40000000

_lock = threading.Lock()
_lib = None


class MatmulDesc(ctypes.Structure):
    """aq_matmul_desc: one matmul of a chain (device pointers as integers)."""
    _fields_ = [("x", ctypes.c_void_p), ("w_packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("y", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("flags", ctypes.c_int64)]


class ChainPlan(ctypes.Structure):
    """aq_chain_plan: filled by aq_chain_prepare, read by aq_chain_run."""
    _fields_ = [("workspace", ctypes.c_void_p), ("count", ctypes.c_int), ("x_bytes", ctypes.c_int),
                ("one_row", ctypes.c_int), ("reserved", ctypes.c_int * 5)]


class AqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where} failed: {status_string(status)}"
        if status == AQ_ERR_CUDA:
            msg += f" ({last_cuda_error()})"
        super().__init__(msg)


def library_path() -> str:
    return LIB


def load() -> ctypes.CDLL:
    """Load libaq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"libaq.so is not built ({LIB}); run __graft_entry__.build()")
            lib = ctypes.CDLL(LIB)
            P, I64, I, U = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint
            lib.aq_matmul_bf16.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, P]
            lib.aq_matmul_bf16.restype = I
            lib.aq_matmul_bf16_ex.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, I, U, P]
            lib.aq_matmul_bf16_ex.restype = I
            lib.aq_quantize_ref.argtypes = [P, I64, I64, I, I, P, P, P]
            lib.aq_quantize_ref.restype = I
            lib.aq_pack_ref.argtypes = [P, I64, I64, I, P]
            lib.aq_pack_ref.restype = I
            lib.aq_status_string.argtypes = [I]
            lib.aq_status_string.restype = ctypes.c_char_p
            lib.aq_last_cuda_error.argtypes = []
            lib.aq_last_cuda_error.restype = ctypes.c_char_p
            lib.aq_chain_workspace_bytes.argtypes = [I]
            lib.aq_chain_workspace_bytes.restype = ctypes.c_size_t
            lib.aq_chain_prepare.argtypes = [ctypes.POINTER(MatmulDesc), I, I, I, P, ctypes.c_size_t,
                                             ctypes.POINTER(ChainPlan)]
            lib.aq_chain_prepare.restype = I
            lib.aq_chain_run.argtypes = [ctypes.POINTER(ChainPlan), P]
            lib.aq_chain_run.restype = I
            lib.aq_chain_run_static.argtypes = [ctypes.POINTER(MatmulDesc), I, I, I, P]
            lib.aq_chain_run_static.restype = I
            lib.aq_read_device_status.argtypes = [P]
            lib.aq_read_device_status.restype = I
            lib.aq_matmul_workspace_bytes.argtypes = [I64, I64]
            lib.aq_matmul_workspace_bytes.restype = ctypes.c_size_t
            lib.aq_matmul_bf16_ws.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, P, ctypes.c_size_t, P]
            lib.aq_matmul_bf16_ws.restype = I
            lib.aq_gather_qmm_workspace_bytes.argtypes = [I64, I64, I64]
            lib.aq_gather_qmm_workspace_bytes.restype = ctypes.c_size_t
            lib.aq_gather_qmm_bf16.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I, I, P,
                                               ctypes.c_size_t, P]
            lib.aq_gather_qmm_bf16.restype = I
            lib.aq_matmul_nvfp4_bf16.argtypes = [P, P, P, ctypes.c_float, P, I64, I64, I64, U, P]
            lib.aq_matmul_nvfp4_bf16.restype = I
            lib.aq_read_probe.argtypes = [P, ctypes.c_size_t, P]
            lib.aq_read_probe.restype = I
            lib.aq_version.argtypes = []
            lib.aq_version.restype = I
            _lib = lib
    return _lib


def declared_functions() -> list[str]:
    """Names of the functions include/aq.h declares."""
    names = []
    for path in sorted(os.listdir(INCLUDE)):
        if path.endswith(".h"):
            text = open(os.path.join(INCLUDE, path)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(aq_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


# ---------------------------------------------------------------- raw C-ABI names

def aq_matmul_bf16(x, w_packed, scales, biases, y, M, N, K, group_size, bits, stream) -> int:
    return load().aq_matmul_bf16(x, w_packed, scales, biases, y, M, N, K, group_size, bits, stream)


def aq_matmul_bf16_ex(x, w_packed, scales, biases, y, M, N, K, group_size, bits, kernel, flags, stream) -> int:
    return load().aq_matmul_bf16_ex(x, w_packed, scales, biases, y, M, N, K, group_size, bits, kernel, flags,
                                    stream)


def aq_quantize_ref(w, N, K, group_size, bits, w_packed, scales_bf16, biases_bf16) -> int:
    return load().aq_quantize_ref(w, N, K, group_size, bits, w_packed, scales_bf16, biases_bf16)


def aq_pack_ref(codes, N, K, bits, w_packed) -> int:
    return load().aq_pack_ref(codes, N, K, bits, w_packed)


def aq_chain_workspace_bytes(count) -> int:
    return load().aq_chain_workspace_bytes(count)


def aq_chain_prepare(descs, count, group_size, bits, workspace, workspace_bytes, plan) -> int:
    return load().aq_chain_prepare(descs, count, group_size, bits, workspace, workspace_bytes, ctypes.byref(plan))


def aq_chain_run(plan, stream) -> int:
    return load().aq_chain_run(ctypes.byref(plan), stream)


def _chain_descs(items, group_size: int, bits: int, independent, release=None):
    """Checks (x, w_packed, scales, biases, y) tensors of a chain and returns
    their aq_matmul_desc array (at least one element).  group_size 16 is an
    NVFP4 chain: (x, w_packed, scales_e4m3 uint8 [N, K/16], global_scale
    float32 [1] on the device, y)."""
    n = len(items)
    if independent is not None and len(independent) != n:
        raise ValueError(f"independent has {len(independent)} flags for {n} matmuls")
    if release is not None and release is not True and len(release) != n:
        raise ValueError(f"release has {len(release)} flags for {n} matmuls")
    arr = (MatmulDesc * max(n, 1))()
    named = []
    for i, (x, w, s, b, y) in enumerate(items):
        if x.dim() != 2 or w.dim() != 2:
            raise ValueError(f"chain item {i}: x and w_packed must be 2-D")
        at = f"chain item {i}: "
        _check(at + "x", x, tuple(x.shape), "bf16")
        if group_size == 16:
            K = x.shape[1]
            blocks_ok = K % 16 == 0          # other K the library rejects itself
            _check(at + "w_packed", w, (None, K // 8 if blocks_ok else None), "word")
            _check(at + "scales_e4m3", s, (w.shape[0], K // 16 if blocks_ok else None), "u8")
            _check(at + "global_scale", b, (1,), "f32")
        else:
            _check_weights(w, s, b, (w.shape[0],), x.shape[1], group_size, bits, prefix=at)
        _check(at + "y", y, (x.shape[0], w.shape[0]), "bf16")
        named += [(at + "x", x), (at + "w_packed", w), (at + "scales", s), (at + "biases", b), (at + "y", y)]
    if n:
        _placed(items[0][0].device, named)
    for i, (x, w, s, b, y) in enumerate(items):
        flags = AQ_CHAIN_INDEPENDENT if (independent and independent[i]) else 0
        if release is True or (release is not None and release[i]):
            flags |= AQ_CHAIN_RELEASE
        arr[i] = MatmulDesc(x.data_ptr(), w.data_ptr(), s.data_ptr(), b.data_ptr(), y.data_ptr(), x.shape[0],
                            w.shape[0], x.shape[1], flags)
    return arr


class Chain:
    """A prepared chain of matmuls over torch CUDA tensors: Chain([(x, w, s, b, y), ...]).run().

    Each y_j is written before matmul j+1 reads its x, so an x may be an
    earlier y.  Holds the device workspace (a torch tensor) and the plan."""

    def __init__(self, items, group_size: int = 64, bits: int = 4, independent=None, release=None):
        import torch

        n = len(items)
        arr = _chain_descs(items, group_size, bits, independent, release)
        self.items = items
        nbytes = aq_chain_workspace_bytes(n)
        dev = items[0][0].device if n else torch.device("cuda")
        self.workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
        self.plan = ChainPlan()
        st = aq_chain_prepare(arr, n, group_size, bits, self.workspace.data_ptr(), nbytes, self.plan)
        if st != AQ_OK:
            raise AqError(st, "aq_chain_prepare")

    def run(self, stream=None):
        import torch

        if stream is None:
            stream = torch.cuda.current_stream()
        st = aq_chain_run(self.plan, stream.cuda_stream)
        if st != AQ_OK:
            raise AqError(st, "aq_chain_run")


def aq_chain_run_static(descs, count, group_size, bits, stream) -> int:
    return load().aq_chain_run_static(descs, count, group_size, bits, stream)


def chain_run_static(items, group_size: int = 64, bits: int = 4, independent=None, stream=None,
                     release=None) -> None:
    """A chain of matmuls over torch CUDA tensors, as Chain(...).run() gives it,
    through the entry point that allocates nothing (aq_chain_run_static; at
    most 256 matmuls).  The tensors are checked as Chain checks them."""
    import torch

    arr = _chain_descs(items, group_size, bits, independent, release)
    if stream is None:
        stream = torch.cuda.current_stream(items[0][0].device) if items else torch.cuda.current_stream()
    st = aq_chain_run_static(arr, len(items), group_size, bits, stream.cuda_stream)
    if st != AQ_OK:
        raise AqError(st, "aq_chain_run_static")


def aq_matmul_workspace_bytes(M, K) -> int:
    return load().aq_matmul_workspace_bytes(M, K)


def aq_matmul_bf16_ws(x, w_packed, scales, biases, y, M, N, K, group_size, bits, workspace, workspace_bytes,
                      stream) -> int:
    return load().aq_matmul_bf16_ws(x, w_packed, scales, biases, y, M, N, K, group_size, bits, workspace,
                                    workspace_bytes, stream)


def aq_gather_qmm_workspace_bytes(R, K, E) -> int:
    return load().aq_gather_qmm_workspace_bytes(R, K, E)


def aq_gather_qmm_bf16(x, w_packed, scales, biases, lhs_indices, rhs_indices, y, R, T, N, K, E, group_size, bits,
                       workspace, workspace_bytes, stream) -> int:
    return load().aq_gather_qmm_bf16(x, w_packed, scales, biases, lhs_indices, rhs_indices, y, R, T, N, K, E,
                                     group_size, bits, workspace, workspace_bytes, stream)


def aq_matmul_nvfp4_bf16(x, w_packed, scales_e4m3, global_scale, y, M, N, K, flags, stream) -> int:
    return load().aq_matmul_nvfp4_bf16(x, w_packed, scales_e4m3, global_scale, y, M, N, K, flags, stream)


def aq_read_probe(buf, nbytes, stream) -> int:
    return load().aq_read_probe(buf, nbytes, stream)


def aq_read_device_status(stream) -> int:
    return load().aq_read_device_status(stream)


def status_string(status: int) -> str:
    return load().aq_status_string(status).decode()


def last_cuda_error() -> str:
    return load().aq_last_cuda_error().decode()


def version() -> int:
    return load().aq_version()


# ---------------------------------------------------------------- torch / numpy helpers

_KERNELS = {"auto": AQ_KERNEL_AUTO, "qmv": AQ_KERNEL_QMV, "qmm": AQ_KERNEL_QMM}


def _kind_ok(t, kind: str) -> bool:
    import torch

    if kind == "bf16":
        return t.dtype == torch.bfloat16
    if kind == "word":   # packed codes: any 32-bit integer type (int32 or uint32)
        return t.element_size() == 4 and not t.is_floating_point() and not t.is_complex()
    if kind == "i32":
        return t.dtype == torch.int32
    if kind == "u8":
        return t.dtype == torch.uint8
    if kind == "f32":
        return t.dtype == torch.float32
    raise AssertionError(kind)


def _check(name: str, t, shape, kind: str) -> None:
    """Raise ValueError unless t has `shape` (None entries are free) and the
    element type `kind`.  The C ABI sees only pointers, so a tensor smaller than
    the shapes say would be read or written out of bounds: the sizes are checked
    here, before any launch."""
    if t.dim() != len(shape) or any(want is not None and int(got) != int(want) for got, want in zip(t.shape, shape)):
        want = "[" + ", ".join("*" if w is None else str(int(w)) for w in shape) + "]"
        raise ValueError(f"{name} has shape {list(t.shape)}, expected {want}")
    if not _kind_ok(t, kind):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {kind}")


def _placed(device, named) -> None:
    """Raise ValueError unless every (name, tensor) is a contiguous CUDA tensor on `device`."""
    for name, t in named:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device}")


def _weight_cols(K: int, group_size: int, bits: int):
    """(code words, groups) per weight row, or (None, None) where K, the group
    size or the code width is one the library itself rejects."""
    if group_size <= 0 or K % group_size or bits not in (4, 8) or (K * bits) % 32:
        return None, None
    return K * bits // 32, K // group_size


def _check_weights(w_packed, scales, biases, lead, K: int, group_size: int, bits: int, prefix: str = "") -> None:
    words, groups = _weight_cols(K, group_size, bits)
    _check(prefix + "w_packed", w_packed, (*lead, words), "word")
    _check(prefix + "scales", scales, (*lead, groups), "bf16")
    _check(prefix + "biases", biases, (*lead, groups), "bf16")


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def matmul(x, w_packed, scales, biases, out=None, *, group_size: int = 64, bits: int = 4,
           kernel: str = "auto", pdl: bool = False, stream=None, flags: int = 0, workspace=None):
    """y = x . dequant(W)^T for torch CUDA tensors (x bf16 [M,K]; w_packed int32/uint32
    [N, K*bits/32]; scales/biases bf16 [N, K/group_size]).  Returns y bf16 [M, N]."""
    import torch

    if x.dim() != 2 or w_packed.dim() != 2:
        raise ValueError("x and w_packed must be 2-D")
    M, K = x.shape
    N = w_packed.shape[0]
    if kernel not in _KERNELS:
        raise ValueError(f"kernel must be one of {sorted(_KERNELS)}")
    _check("x", x, (M, K), "bf16")
    _check_weights(w_packed, scales, biases, (N,), K, group_size, bits)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check("out", out, (M, N), "bf16")
    named = [("x", x), ("w_packed", w_packed), ("scales", scales), ("biases", biases), ("out", out)]
    if workspace is not None:
        if kernel != "auto" or pdl or flags:
            raise ValueError("a workspace goes with the default kernel choice and no flags")
        _check("workspace", workspace, (None,), "u8")
        named.append(("workspace", workspace))
    _placed(x.device, named)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    if workspace is not None:
        where = "aq_matmul_bf16_ws"
        st = aq_matmul_bf16_ws(x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(), biases.data_ptr(),
                               out.data_ptr(), M, N, K, group_size, bits, workspace.data_ptr(), _nbytes(workspace),
                               stream.cuda_stream)
    else:
        where = "aq_matmul_bf16_ex"
        st = aq_matmul_bf16_ex(x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(), biases.data_ptr(),
                               out.data_ptr(), M, N, K, group_size, bits, _KERNELS[kernel],
                               (AQ_FLAG_PDL if pdl else 0) | flags, stream.cuda_stream)
    if st != AQ_OK:
        raise AqError(st, where)
    return out


def quantize_ref(w, group_size: int = 64, bits: int = 4):
    """Host min-max quantization of a float32 numpy array [N, K] (library's aq_quantize_ref)."""
    import numpy as np

    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    wp = np.empty((N, K * bits // 32), np.uint32)
    s = np.empty((N, K // group_size), np.uint16)
    b = np.empty((N, K // group_size), np.uint16)
    st = aq_quantize_ref(w.ctypes.data, N, K, group_size, bits, wp.ctypes.data, s.ctypes.data, b.ctypes.data)
    if st != AQ_OK:
        raise AqError(st, "aq_quantize_ref")
    return wp, s, b


def pack_ref(codes, bits: int = 4):
    """Host packing of uint8 codes [N, K] (library's aq_pack_ref)."""
    import numpy as np

    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = codes.shape
    wp = np.empty((N, K * bits // 32), np.uint32)
    st = aq_pack_ref(codes.ctypes.data, N, K, bits, wp.ctypes.data)
    if st != AQ_OK:
        raise AqError(st, "aq_pack_ref")
    return wp


def gather_qmm(x, w_packed, scales, biases, lhs_indices, rhs_indices, out=None, workspace=None, *,
               group_size: int = 64, bits: int = 4, stream=None):
    """Expert-indexed matmul for torch CUDA tensors: x bf16 [T, K]; w_packed int32
    [E, N, K*bits/32]; scales/biases bf16 [E, N, K/group_size]; lhs/rhs int32 [R]
    (rhs non-decreasing).  Returns y bf16 [R, N]; allocates the workspace if none
    is given (a uint8 CUDA tensor of aq_gather_qmm_workspace_bytes)."""
    import torch

    if x.dim() != 2 or w_packed.dim() != 3 or lhs_indices.dim() != 1:
        raise ValueError("x must be 2-D, w_packed 3-D and lhs_indices 1-D")
    T, K = x.shape
    E, N = w_packed.shape[0], w_packed.shape[1]
    R = lhs_indices.shape[0]
    _check("x", x, (T, K), "bf16")
    _check_weights(w_packed, scales, biases, (E, N), K, group_size, bits)
    _check("lhs_indices", lhs_indices, (R,), "i32")
    _check("rhs_indices", rhs_indices, (R,), "i32")
    if out is None:
        out = torch.empty((R, N), dtype=torch.bfloat16, device=x.device)
    _check("out", out, (R, N), "bf16")
    if workspace is not None:
        _check("workspace", workspace, (None,), "u8")
    _placed(x.device, [("x", x), ("w_packed", w_packed), ("scales", scales), ("biases", biases),
                       ("lhs_indices", lhs_indices), ("rhs_indices", rhs_indices), ("out", out)]
            + ([("workspace", workspace)] if workspace is not None else []))
    if workspace is None:
        need = aq_gather_qmm_workspace_bytes(R, K, E)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    st = aq_gather_qmm_bf16(x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(), biases.data_ptr(),
                            lhs_indices.data_ptr(), rhs_indices.data_ptr(), out.data_ptr(), R, T, N, K, E,
                            group_size, bits, workspace.data_ptr(), _nbytes(workspace), stream.cuda_stream)
    if st != AQ_OK:
        raise AqError(st, "aq_gather_qmm_bf16")
    return out


def matmul_nvfp4(x, w_packed, scales_e4m3, global_scale: float = 1.0, out=None, *, pdl: bool = False, stream=None):
    """NVFP4 decode matmul for torch CUDA tensors: x bf16 [M, K]; w_packed int32
    [N, K/8] (E2M1 codes); scales_e4m3 uint8 [N, K/16].  Returns y bf16 [M, N]."""
    import torch

    if x.dim() != 2 or w_packed.dim() != 2:
        raise ValueError("x and w_packed must be 2-D")
    M, K = x.shape
    N = w_packed.shape[0]
    _check("x", x, (M, K), "bf16")
    blocks_ok = K % 16 == 0          # other K the library rejects itself
    _check("w_packed", w_packed, (N, K // 8 if blocks_ok else None), "word")
    _check("scales_e4m3", scales_e4m3, (N, K // 16 if blocks_ok else None), "u8")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check("out", out, (M, N), "bf16")
    _placed(x.device, [("x", x), ("w_packed", w_packed), ("scales_e4m3", scales_e4m3), ("out", out)])
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    st = aq_matmul_nvfp4_bf16(x.data_ptr(), w_packed.data_ptr(), scales_e4m3.data_ptr(), float(global_scale),
                              out.data_ptr(), M, N, K, AQ_FLAG_PDL if pdl else 0, stream.cuda_stream)
    if st != AQ_OK:
        raise AqError(st, "aq_matmul_nvfp4_bf16")
    return out
