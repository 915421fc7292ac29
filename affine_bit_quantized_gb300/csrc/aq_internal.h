// Internal declarations shared by the libaq translation units (not installed).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "aq.h"

namespace aq {

// Arguments of one y = x . dequant(W)^T launch, already validated.
struct MatmulArgs {
    const void *x;           // bf16 [M, K]
    const uint32_t *w;       // uint32 [N, K*bits/32]
    const uint16_t *scales;  // bf16 bits [N, K/64]
    const uint16_t *biases;  // bf16 bits [N, K/64]
    void *y;                 // bf16 [M, N]
    int64_t M, N, K;
    bool pdl;                // launch with programmatic stream serialization
    cudaStream_t stream;
    int *status;             // device status word (bounded waits record timeouts here)
    uint64_t timeout_ns;     // deadline of every bounded device-side wait
    bool debug_skip_copy;    // test hook: the kernel's producer leaves out one copy
    int bits = 4;            // code width: 4 or 8
    void *xf16 = nullptr;    // tensor-core path: M*K*2 bytes of caller workspace for x converted once
    bool split_rows = false; // TMA-fed decode kernel: CTA pairs take the two halves of x's rows
};

// Values of the device status word.
constexpr int AQ_DEVICE_STATUS_OK = 0;
constexpr int AQ_DEVICE_STATUS_TIMEOUT = 5;
constexpr int AQ_DEVICE_STATUS_BAD_INDEX = 6;

// Weight-streaming kernel for up to 16 rows of x (qmv.cu).  Requires
// 1 <= M <= 16, N >= 1, K >= 64.
cudaError_t launch_qmv(const MatmulArgs &a);

// TMA-fed weight-streaming kernel (qmv_tma.cu) for 1 <= M <= 8, K % 512 == 0
// and 16-byte aligned scales/biases (x beyond 32 KB: K in passes).
// the driver's tensor-map encoder (null if the driver does not offer it)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// tensor map of packed codes for the decode kernels: a stage (32 rows x 1024 bytes) per copy
bool encode_codes_3d(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows);
bool qmv_tma_supported(const MatmulArgs &a);
int qmv_tma_passes(const MatmulArgs &a);   // K passes the TMA kernel makes (x staged per pass)
bool qmv_tma_preferred(const MatmulArgs &a);   // faster than the general kernel for this 4-bit shape
cudaError_t launch_qmv_tma(const MatmulArgs &a);

// Tensor-core kernel (qmm.cu) for any M >= 1 with K % 512 == 0 and 16-byte
// aligned scales/biases.
bool qmm_supported(const MatmulArgs &a);
cudaError_t launch_qmm(const MatmulArgs &a);

// Expert-indexed matmul (qmm.cu): row r of y = x[lhs[r]] . dequant(W[rhs[r]])^T,
// rows grouped by expert (rhs non-decreasing), through a plan and a gathered
// copy of x in the caller's workspace and the tensor-core kernel.
constexpr int kMaxExperts = 1024;
struct GatherArgs {
    const void *x;           // bf16 [T, K]
    const uint32_t *w;       // uint32 [E, N, K*bits/32]
    const uint16_t *scales;  // bf16 bits [E, N, K/64]
    const uint16_t *biases;  // bf16 bits [E, N, K/64]
    const int *lhs, *rhs;    // int32 [R]
    void *y;                 // bf16 [R, N]
    int64_t R, T, N, K, E;
    int bits;
    void *workspace;         // gather_workspace_bytes(R, K, E), 128-byte aligned
    cudaStream_t stream;
    int *status;
    uint64_t timeout_ns;
};
size_t gather_workspace_bytes(int64_t R, int64_t K, int64_t E);
cudaError_t launch_gather_qmm(const GatherArgs &g);

// NVFP4 weight-streaming kernel (nvfp4_qmv.cu): 1 <= M <= 8, K % 256 == 0,
// M*K <= 16384, 16-byte aligned x, codes and scales.
struct Nvfp4Args {
    const void *x;            // bf16 [M, K]
    const uint32_t *w;        // FP4 E2M1 codes [N, K/8]
    const uint8_t *scales;    // FP8 E4M3 [N, K/16]
    float global_scale;
    void *y;                  // bf16 [M, N]
    int64_t M, N, K;
    bool pdl;
    cudaStream_t stream;
    int *status;
    uint64_t timeout_ns;
    int rows = 0;             // rows of x per CTA: groups of CTAs split M and walk the same tiles (0: M)
};
cudaError_t launch_nvfp4_qmv(const Nvfp4Args &a);

// Chains of decode matmuls in one persistent launch (qmv_chain.cu).
size_t chain_workspace_bytes(int count);
aq_status chain_prepare(const aq_matmul_desc *descs, int count, int group_size, int bits, void *workspace,
                        size_t workspace_bytes, aq_chain_plan *plan, cudaError_t *err);
cudaError_t chain_run(const aq_chain_plan *plan, uint64_t timeout_ns, int *status, cudaStream_t stream);
// The allocation-free variant: plan and counters in a static device array.
int chain_static_max();
aq_status chain_run_static(const aq_matmul_desc *descs, int count, int group_size, int bits, uint64_t timeout_ns,
                           int *status, cudaStream_t stream, cudaError_t *err);

// Read-only TMA stream over floor(bytes / 16384) chunks of 16 KB (read_probe.cu).
cudaError_t launch_read_probe(const void *buf, size_t bytes, uint64_t timeout_ns, int *status, cudaStream_t stream);

}  // namespace aq
