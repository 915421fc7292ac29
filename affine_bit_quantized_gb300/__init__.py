"""Affine group-quantized matmul for NVIDIA GB300 (sm_103a).

y[M,N] = x[M,K] . dequant(W)^T with W stored as 4-bit codes packed eight per
uint32 (lowest nibble = lowest k) and one bf16 scale and bias per group of 64
along K.  The work runs in libaq.so (hand-written CUDA); this package is a thin
ctypes binding with the C ABI's names.
"""
from ._lib import (AQ_CHAIN_DEBUG_SKIP_COPY, AQ_CHAIN_INDEPENDENT, AQ_CHAIN_RELEASE, AQ_ERR_ALIGNMENT, AQ_ERR_BAD_INDEX, AQ_ERR_CUDA, AQ_ERR_INVALID_ARG, AQ_ERR_TIMEOUT, AQ_ERR_UNSUPPORTED,
                   AQ_FLAG_DEBUG_SKIP_COPY, AQ_FLAG_PDL, AQ_KERNEL_AUTO, AQ_KERNEL_QMM, AQ_KERNEL_QMV, AQ_OK, AqError, Chain, ChainPlan, MatmulDesc, chain_run_static, aq_chain_prepare, aq_chain_run, aq_chain_run_static,
                   aq_chain_workspace_bytes, aq_gather_qmm_bf16, aq_gather_qmm_workspace_bytes, aq_matmul_bf16, aq_matmul_bf16_ws, aq_matmul_nvfp4_bf16, aq_matmul_workspace_bytes,
                   aq_matmul_bf16_ex, aq_pack_ref, aq_quantize_ref, aq_read_device_status, aq_read_probe, declared_functions, last_cuda_error,
                   gather_qmm, library_path, load, matmul, matmul_nvfp4, pack_ref, quantize_ref, status_string, version)

__all__ = [n for n in dir() if not n.startswith("_")]
