/*
 * aq.h -- C ABI of libaq, the affine group-quantized matmul for NVIDIA GB300
 * (sm_103a).
 *
 * The operation is the one the "MLX CUDA Cleanup Plan" page asks a
 * backend-neutral accelerator call to provide: bf16 activations times weights
 * packed into 32-bit words with bf16 scales and biases (Target Architecture,
 * sections 1-2), in the 4-bit, group-size-64 affine packed form of its
 * Refactor Plan, Phase 3:
 *
 *     y[m,n] = sum_k x[m,k] * w[n,k],   w[n,k] = scale[n,k/64] * q[n,k] + bias[n,k/64]
 *
 *   x        bf16 [M, K], row-major.
 *   w_packed uint32 [N, K/8]: the 4-bit unsigned codes q[n, 0..K), eight per
 *            word, the lowest nibble holding the lowest k.
 *   scales   bf16 [N, K/64], row-major; biases likewise.
 *   y        bf16 [M, N], row-major; each element is the fp32-accumulated sum
 *            rounded to nearest-even bf16.
 *
 * Decode on the pages is bound by streaming these weights ("epic: CUDA (MLX
 * backend) prefill and decode acceleration program", Diagnosis; "gemma-4
 * decode carries ~44 ms/token ...", re-scope paragraph), so M = 1..16 runs a
 * weight-streaming kernel and larger M a tensor-core GEMM.
 *
 * Conventions shared by every entry point below:
 *  - Ownership: the caller owns every buffer and the stream.  No entry point
 *    allocates or frees device memory, and none synchronizes the host (the
 *    Hard Constraints section of the cleanup plan: no extra copies, staging
 *    buffers or synchronization points on the hot path), apart from the
 *    exceptions stated at aq_chain_prepare, aq_chain_run_static and
 *    aq_read_device_status.  The library's own device memory is two
 *    file-scope arrays that every GPU loading it holds until the process
 *    exits: a 4-byte status word (aq_read_device_status) and the 132 KB
 *    scratch of aq_chain_run_static.
 *  - Device pointers are plain CUDA device addresses of the current device.
 *    `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - Work is enqueued asynchronously on `stream`; an AQ_OK return means the
 *    arguments were valid and the launch was accepted, not that it finished.
 *  - Arguments are validated before anything is enqueued; on any error
 *    nothing is launched and the output is left untouched.
 *  - Thread safety: every entry point may be called from several host threads
 *    at once.  aq_last_cuda_error() is per host thread.
 */
#ifndef AQ_H
#define AQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum aq_status {
    AQ_OK = 0,
    AQ_ERR_INVALID_ARG = 1, /* negative size, null pointer, K not a multiple of the group size */
    AQ_ERR_UNSUPPORTED = 2, /* bits or group_size outside what this build implements */
    AQ_ERR_ALIGNMENT = 3,   /* a pointer without the alignment stated below */
    AQ_ERR_CUDA = 4,        /* the CUDA runtime refused the launch: see aq_last_cuda_error() */
    AQ_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (see aq_read_device_status) */
    AQ_ERR_BAD_INDEX = 6    /* aq_gather_qmm_bf16 met an index out of range or experts out of
                               order (see aq_read_device_status) */
} aq_status;

/* Kernel choice for aq_matmul_bf16_ex.  AUTO picks by M exactly as
 * aq_matmul_bf16 does. */
typedef enum aq_kernel {
    AQ_KERNEL_AUTO = 0,
    AQ_KERNEL_QMV = 1, /* weight-streaming decode kernels, any M.  The TMA-fed kernel
                          wherever it applies (K % 512 == 0, 16-byte aligned scales and
                          biases; up to 16 rows of x per launch, W streamed once per
                          launch), else the general one in launches of 16 rows of x (both
                          code widths).  AQ_KERNEL_AUTO chooses among these (and the GEMM
                          kernel above 16 rows) by measured speed; for 9..16 rows whose x
                          needs several K passes (4-bit codes: over at least one 32-row
                          tile per SM) it runs the TMA-fed kernel once, with pairs of CTAs
                          that take the two halves of the rows and walk the same tiles of
                          W together. */
    AQ_KERNEL_QMM = 2  /* tensor-core GEMM kernel (tcgen05); any M >= 1 */
} aq_kernel;

/* Flags for aq_matmul_bf16_ex (bits of its unsigned `flags`; macros, because
 * bit 31 is outside the range ISO C allows an enumerator). */
/* Launch with programmatic dependent launch: the kernel may start while
 * the previous kernel on the stream is still running and begins streaming
 * w_packed/scales/biases before it waits for that kernel to finish.  It
 * reads x and writes y only after the wait.  PRECONDITION: the weights
 * were not written by the kernel immediately before on the stream. */
#define AQ_FLAG_PDL 0x1u
/* Test hook for the failure path of the bounded device-side waits: the
 * kernel's copy producer leaves out one of its copies, so the consumers'
 * wait for it expires (after 20 ms instead of the normal 2 s), the kernel
 * records a timeout in the device status word and returns without a valid y.
 * Taken by the weight-streaming kernel (1 <= M <= 8, K a multiple of 512,
 * 16-byte aligned scales and biases) and by the tensor-core kernel
 * (AQ_KERNEL_QMM); elsewhere AQ_ERR_UNSUPPORTED.  Read the outcome with
 * aq_read_device_status(). */
#define AQ_FLAG_DEBUG_SKIP_COPY 0x80000000u

/*
 * y = x . dequant(W)^T as defined above.
 *
 *   M, N, K     M >= 0, N >= 0, K >= 0; K a multiple of group_size.  M == 0 or
 *               N == 0 launches nothing and returns AQ_OK; K == 0 writes y = 0.
 *   group_size  64.  Other values return AQ_ERR_UNSUPPORTED.
 *   bits        4 or 8.  Other values return AQ_ERR_UNSUPPORTED.  8-bit codes
 *               need 16-byte aligned scales and biases (AQ_ERR_ALIGNMENT
 *               otherwise).  With K not a multiple of 512 (either width) the
 *               TMA-fed and tensor-core kernels do not apply and every M runs
 *               on the general decode kernel, in launches of 16 rows of x that
 *               each stream W: correct, but slow for large M.
 *   Alignment   x and w_packed 16-byte aligned; scales, biases and y 2-byte
 *               aligned; otherwise AQ_ERR_ALIGNMENT.
 *   Aliasing    y must not overlap any input.
 *   Numerics    fp32 accumulation, one rounding to bf16 per output.  Inputs
 *               with NaN or Inf propagate them.  The tensor-core path
 *               (M > 16) converts x to fp16 on chip: it needs |x| <= 65504,
 *               and |x| below 2^-14 loses relative precision (not its
 *               contribution to y, which stays far below one bf16 ulp for
 *               weights of unit scale or less).
 *   Result is deterministic: the same inputs give the same bits on every
 *   call (fixed reduction order, no floating-point atomics).
 */
aq_status aq_matmul_bf16(const void *x, const uint32_t *w_packed, const void *scales,
                         const void *biases, void *y, int64_t M, int64_t N, int64_t K,
                         int group_size, int bits, void *stream);

/* As aq_matmul_bf16, with an explicit kernel choice (aq_kernel) and flags
 * (AQ_FLAG_*).  Unknown kernel values or flag bits return AQ_ERR_INVALID_ARG. */
aq_status aq_matmul_bf16_ex(const void *x, const uint32_t *w_packed, const void *scales,
                            const void *biases, void *y, int64_t M, int64_t N, int64_t K,
                            int group_size, int bits, int kernel, unsigned flags, void *stream);

/*
 * Host utility (test data): min-max affine quantization of float weights
 * w[N, K] (host memory) into the packed format above.  The pages give no
 * quantization procedure; this one takes, per group, scale = (max - min) /
 * (2^bits - 1) and bias = min, each rounded to nearest-even bf16, then
 * q = clamp(round_half_even((w - bias) / scale), 0, 2^bits - 1) with the
 * rounded scale and bias (a constant group gets scale 0 and q = 0).
 * Outputs are host buffers of N*K*bits/32 words and N*K/group_size bf16 bit
 * patterns each.  bits 4 or 8; K a multiple of group_size (> 0).  Runs
 * synchronously on the calling thread.
 */
aq_status aq_quantize_ref(const float *w, int64_t N, int64_t K, int group_size, int bits,
                          uint32_t *w_packed, uint16_t *scales_bf16, uint16_t *biases_bf16);

/* Host utility: pack codes[N, K] (host, one code per byte, values below
 * 2^bits) into words as described above.  bits 4 or 8; K a multiple of
 * 32/bits.  A code >= 2^bits returns AQ_ERR_INVALID_ARG. */
aq_status aq_pack_ref(const uint8_t *codes, int64_t N, int64_t K, int bits, uint32_t *w_packed);

/*
 * Chains of decode matmuls in one launch.
 *
 * A decode step is a sequence of matmuls, each reading an x produced by
 * earlier work; its cost is streaming the weights ("gemma-4 decode carries
 * ~44 ms/token ...", re-scope paragraph), and the "MLX CUDA Cleanup Plan"
 * page (Refactor Plan, Phase 5) asks for a device-resident step with
 * persistent work buffers.  aq_chain_run executes count matmuls in order in a
 * single persistent kernel: matmul j reads its x only after every earlier
 * matmul of the chain has written all of its y (so x_j may be an earlier
 * y_i), unless it is flagged AQ_CHAIN_INDEPENDENT, while the weights of the
 * next matmuls keep streaming.  So w_packed, scales and biases must not be
 * written by any matmul of the chain (they are read ahead of the ordering).
 *
 * Each descriptor follows aq_matmul_bf16's definition, with the limits of the
 * weight-streaming kernel: 1 <= M <= 8, K a multiple of 512, M*K <= 16384
 * (K rounded up to 2048 codes for 4-bit codes, 1024 for 8-bit), x, w_packed,
 * scales and biases 16-byte aligned, y 2-byte aligned.
 *
 * NVFP4 chains (group_size 16, bits 4): every matmul follows
 * aq_matmul_nvfp4_bf16's definition; `scales` is then the uint8 [N, K/16]
 * E4M3 block scales and `biases` the device address of the tensor's fp32
 * global scale (one float, 4-byte aligned, read by the kernel at run time).
 * Limits: 1 <= M <= 8, K a multiple of 256, M*K <= 16384 (K rounded up to
 * 2048), x, w_packed and scales 16-byte aligned.  A chain holds one format.
 */
typedef struct aq_matmul_desc {
    const void *x;            /* bf16 [M, K], device */
    const uint32_t *w_packed; /* uint32 [N, K/8], device */
    const void *scales;       /* bf16 [N, K/64], device (NVFP4: uint8 E4M3 [N, K/16]) */
    const void *biases;       /* bf16 [N, K/64], device (NVFP4: const float *, the global scale) */
    void *y;                  /* bf16 [M, N], device, written */
    int64_t M, N, K;
    int64_t flags;            /* 0 or AQ_CHAIN_INDEPENDENT | AQ_CHAIN_RELEASE; AQ_CHAIN_DEBUG_SKIP_COPY (test hook) */
} aq_matmul_desc;

enum {
    /* This matmul does not read the output of the matmul before it in the
     * chain (e.g. k and v after q, or up after gate: same input, no mutual
     * dependency).  It is ordered after whatever the previous matmul waited
     * for, but not after the previous matmul itself, so the two overlap.  A
     * run of matmuls on the same x buffer with this flag loads x once. */
    AQ_CHAIN_INDEPENDENT = 1,
    /* Publish the completion of this matmul's dependency group with a
     * GPU-scope release even where no later matmul of the chain needs it.
     * aq_chain_prepare releases a group's completion (a memory fence that
     * waits for the group's y stores to reach L2, about 0.9 us on GB300)
     * only where a later matmul reads or rewrites memory that a matmul up to
     * that group wrote, or rewrites memory one of them read (checked on the
     * byte ranges of every x, w_packed, scales, biases and y); elsewhere the
     * next group still starts only after every tile of the previous one is
     * stored, without the fence.  All outputs are visible to work that
     * follows the launch on the stream either way.  This flag forces the
     * fence (measurement, or callers with their own reasons). */
    AQ_CHAIN_RELEASE = 2,
    /* Test hook for the failure path of the chain's bounded waits: the first
     * CTA's producer leaves out the first copy of this matmul's weights, so
     * waits in the kernel expire (after 20 ms instead of 2 s), a timeout is
     * recorded in the device status word (read it with
     * aq_read_device_status()) and the outputs of the run are not valid. */
    AQ_CHAIN_DEBUG_SKIP_COPY = 0x40000000
};

/* Filled by aq_chain_prepare; owned by the caller, read by aq_chain_run. */
typedef struct aq_chain_plan {
    void *workspace; /* the caller's device workspace (plan records + counters) */
    int count;       /* number of matmuls */
    int x_bytes;     /* largest M*K*2 of the chain */
    int one_row;     /* 1 if every matmul has M == 1 */
    int reserved[5];  /* internal; reserved[3]: dependency groups whose completion is released */
} aq_chain_plan;

/* Device workspace bytes a chain of `count` matmuls needs (one 512-byte
 * record per matmul plus 4 bytes of completion counter per matmul, rounded
 * up to 128). */
size_t aq_chain_workspace_bytes(int count);

/* Set-up call: validates the descriptors, encodes one record per matmul
 * (TMA descriptors, pointers, sizes) and copies them into `workspace`
 * (device memory, 128-byte aligned, at least aq_chain_workspace_bytes(count)
 * bytes, owned by the caller and left untouched by anything else until the
 * last aq_chain_run with this plan has finished).  This call synchronizes (it
 * copies the records with cudaMemcpy); the pointers it records are used by
 * every later run.  Errors: AQ_ERR_INVALID_ARG (bad sizes, null pointers,
 * small workspace), AQ_ERR_UNSUPPORTED (outside the limits above or bits/group
 * size), AQ_ERR_ALIGNMENT, AQ_ERR_CUDA.  count == 0 gives an empty plan. */
aq_status aq_chain_prepare(const aq_matmul_desc *descs, int count, int group_size, int bits,
                           void *workspace, size_t workspace_bytes, aq_chain_plan *plan);

/* Enqueues the chain on `stream`: a reset of the completion counters
 * (cudaMemsetAsync on the workspace) and one cooperative launch of the
 * persistent kernel.  Asynchronous; allocates nothing.  Runs that overlap on
 * the GPU must use different workspaces.  A bounded wait that expires inside
 * the kernel is reported by aq_read_device_status(). */
aq_status aq_chain_run(const aq_chain_plan *plan, void *stream);

/*
 * aq_chain_run as a single call that allocates nothing, for callers that
 * cannot hand this library any device memory: a plugin inside a host
 * framework that owns the whole device memory pool and gives plugins no
 * workspace, or a serving loop that must not reach an allocator after
 * start-up (an allocation can synchronize the device, and can fail once
 * memory is fragmented).  An addition of this library, not a call the pages
 * describe.
 *
 * Same descriptors, semantics and limits as aq_chain_prepare + aq_chain_run,
 * at most 256 matmuls per call (a longer chain returns AQ_ERR_INVALID_ARG and
 * launches nothing).  The plan records and completion counters live in a
 * static device array of 132 KB that every GPU loading this library holds
 * until the process exits; the caller still owns every input and output
 * buffer.  Each call encodes the descriptors again, copies them into that
 * array on `stream` (cudaMemcpyAsync from a static host array in pageable
 * memory) and clears the counters before its launch.  Because the copy is
 * from pageable memory, the call may wait, before it returns, until the
 * stream's earlier work has finished.  Calls from several host threads are
 * serialized inside the library (copy, clear and launch of one call reach
 * the stream together).  All calls share the array: calls whose work
 * overlaps on the GPU (other streams, or another device-side user of the
 * same array) race, so serialize them.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) and should come before
 * any stream capture.  Calls no cudaMalloc or cudaFree.
 */
aq_status aq_chain_run_static(const aq_matmul_desc *descs, int count, int group_size, int bits,
                              void *stream);

/* Static, NUL-terminated name of a status code. */
const char *aq_status_string(aq_status status);

/* Workspace with which aq_matmul_bf16_ws converts x once for the tensor-core
 * kernel: M*K*2 bytes where that kernel is taken (M > 16), else 0. */
size_t aq_matmul_workspace_bytes(int64_t M, int64_t K);

/* aq_matmul_bf16 with a caller workspace (device, 128-byte aligned, owned by
 * the caller, at least aq_matmul_workspace_bytes(M, K) bytes): on the
 * tensor-core path x is converted to fp16 once into the workspace (one extra
 * launch) and copied by TMA straight into the MMA operand tiles, instead of
 * every CTA converting its x tiles again; the results are bit-identical to
 * aq_matmul_bf16's.  A null or smaller workspace gives aq_matmul_bf16's path.
 * Other arguments, errors and numerics as aq_matmul_bf16. */
aq_status aq_matmul_bf16_ws(const void *x, const uint32_t *w_packed, const void *scales,
                            const void *biases, void *y, int64_t M, int64_t N, int64_t K,
                            int group_size, int bits, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * Expert-indexed matmul for mixture-of-experts prefill: MLX's gather_qmm with
 * transposed weights, the grouped-GEMM path behind the MoE prefill gap of
 * "epic: CUDA (MLX backend) prefill and decode acceleration program"
 * (Diagnosis table, MoE prefill row; Phase 3).  For r in [0, R):
 *
 *     y[r, :] = x[lhs_indices[r], :] . dequant(W_e)^T,   e = rhs_indices[r]
 *
 * with W_e, its scales and biases the e-th of E matrices stacked in
 * w_packed [E, N, K*bits/32], scales and biases [E, N, K/group_size], each as
 * in aq_matmul_bf16.
 *
 *   x            bf16 [T, K], device; lhs_indices int32 [R], device, in [0, T)
 *   rhs_indices  int32 [R], device, in [0, E) and non-decreasing: the rows of
 *                an expert are contiguous (sort the (token, expert) pairs by
 *                expert first, as a MoE layer does before its experts)
 *   y            bf16 [R, N], device, written
 *   R >= 0 (0 launches nothing), T >= 1, N >= 1, 1 <= E <= 1024,
 *   K a multiple of 512; group_size 64; bits 4 or 8.
 *   workspace    device, 128-byte aligned, at least
 *                aq_gather_qmm_workspace_bytes(R, K, E) bytes, owned by the
 *                caller (the work plan, and x's rows in row order converted to
 *                fp16 for the tensor cores: R*K*2 bytes)
 *   Alignment    x, w_packed, scales, biases 16-byte aligned; indices 4-byte;
 *                y 2-byte (AQ_ERR_ALIGNMENT otherwise).
 * Runs as three launches on `stream`: a plan of the work tiles per expert
 * (which also checks the indices), the gather of x's rows, and the
 * tensor-core kernel over the tiles.  Indices out of range or out of order
 * are reported by aq_read_device_status() as AQ_ERR_BAD_INDEX and y is not
 * written.  Numerics as aq_matmul_bf16's tensor-core path (|x| < 65504).
 * Asynchronous; allocates nothing; deterministic.
 */
size_t aq_gather_qmm_workspace_bytes(int64_t R, int64_t K, int64_t E);
aq_status aq_gather_qmm_bf16(const void *x, const uint32_t *w_packed, const void *scales,
                             const void *biases, const int32_t *lhs_indices,
                             const int32_t *rhs_indices, void *y, int64_t R, int64_t T,
                             int64_t N, int64_t K, int64_t E, int group_size, int bits,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * NVFP4 decode matmul ("MLX CUDA Cleanup Plan", Refactor Plan, Phase 3b: the
 * mode=nvfp4, group_size=16 checkpoint and a CUDA NVFP4 qmv kept separate
 * from the affine path):
 *
 *     y[m, n] = sum_k x[m, k] * global_scale * e4m3(scales[n, k/16]) * e2m1(q[n, k])
 *
 *   x             bf16 [M, K], device
 *   w_packed      uint32 [N, K/8], device: FP4 E2M1 codes (bit 3 sign, two
 *                 exponent bits with bias 1, one mantissa bit), eight per word,
 *                 lowest nibble = lowest k
 *   scales_e4m3   uint8 [N, K/16], device: FP8 E4M3 block scales (no
 *                 infinities; S.1111.111 is NaN and propagates)
 *   global_scale  the tensor's fp32 scale (1.0f if it has none)
 *   y             bf16 [M, N], device, written; fp32 accumulation, one rounding
 *   M >= 0, N >= 1, K a multiple of 256 up to 32768 (M == 0 or N == 0:
 *   nothing launched).  Each CTA takes up to r = min(8, 32768 / K) rows of x;
 *   one launch takes up to 8 r rows on groups of CTAs that split them and walk
 *   the same tiles of W together (W read from DRAM about once per launch).
 *   x, w_packed and scales_e4m3 16-byte aligned,
 *   y 2-byte aligned.  Errors: AQ_ERR_INVALID_ARG, AQ_ERR_UNSUPPORTED (sizes
 *   outside these limits), AQ_ERR_ALIGNMENT, AQ_ERR_CUDA.  Asynchronous;
 *   allocates nothing; deterministic.  AQ_FLAG_PDL is accepted in `flags`.
 */
aq_status aq_matmul_nvfp4_bf16(const void *x, const uint32_t *w_packed, const uint8_t *scales_e4m3,
                               float global_scale, void *y, int64_t M, int64_t N, int64_t K,
                               unsigned flags, void *stream);

/* Text of the last CUDA runtime error seen by an entry point on this host
 * thread ("" if none).  Valid until the next call on this thread. */
const char *aq_last_cuda_error(void);

/* Waits for `stream` to finish, then reads and clears the library's device
 * status word on the current device: AQ_ERR_TIMEOUT if a bounded wait inside
 * a kernel expired since the last read (that kernel's output is then not
 * valid), AQ_ERR_BAD_INDEX if an aq_gather_qmm_bf16 call found invalid
 * indices (it then wrote nothing to y), else AQ_OK; AQ_ERR_CUDA if the
 * synchronization or copy failed.
 * A debugging call: it synchronizes the host with the stream. */
aq_status aq_read_device_status(void *stream);

/*
 * Measurement probe, not an operation of the pages (they have no counterpart;
 * their roofline is bytes per token over the memory bandwidth, "epic: CUDA
 * (MLX backend) prefill and decode acceleration program", Diagnosis).  Reads
 * floor(bytes / 16384) * 16384 bytes of `buf` (device, 16-byte aligned,
 * bytes >= 16384) once, with the same TMA bulk copies into shared memory that
 * the weight-streaming kernels use and no arithmetic: one persistent CTA per
 * SM, twelve 16 KB copies in flight each.  Time it on `stream` to get the
 * device's read-only streaming rate, the ceiling of a kernel that only reads.
 * Asynchronous; allocates nothing; writes no memory.  AQ_ERR_INVALID_ARG for a
 * null or too small buffer, AQ_ERR_ALIGNMENT, AQ_ERR_CUDA.
 */
aq_status aq_read_probe(const void *buf, size_t bytes, void *stream);

/* Library version, major*10000 + minor*100 + patch. */
int aq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AQ_H */
