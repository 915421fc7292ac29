// A chain of decode matmuls in one persistent launch.
//
// A decode step is a sequence of y_j = x_j . dequant(W_j)^T where x_j depends
// on earlier outputs, and the pages trace the step's cost to streaming the
// weights ("gemma-4 decode carries ~44 ms/token ...", re-scope paragraph) and
// ask for a device-resident step with persistent work buffers and no host
// round trips ("MLX CUDA Cleanup Plan", Refactor Plan Phase 5).  Launching one
// kernel per matmul pays a launch and a full drain / refill of the weight
// stream at every dependency.  This kernel instead runs the whole chain:
//
//  * CTAs are persistent and co-resident (cooperative launch), with the same
//    producer / consumer structure and arithmetic as the single-matmul
//    TMA kernel (qmv_tma.cu): 16-row x 2048-code stages through a 4-stage
//    shared-memory ring, mma.sync on exact 128 + q bf16 codes, per-group fold;
//  * the producer walks the matmuls in order and keeps streaming the NEXT
//    matmuls' weights while the consumers wait for a dependency, because
//    weights never depend on earlier outputs;
//  * matmul j reads its x only after every CTA has stored all of its tiles of
//    matmul j-1 (a completion counter per matmul in the caller's workspace,
//    release / acquire at GPU scope, bounded wait), which is the same
//    ordering a chain of stream-ordered launches gives.
//
// The plan (one record per matmul: three TMA descriptors plus pointers and
// sizes) and the counters live in caller-owned device memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "aq.h"
#include "aq_internal.h"
#include "aq_ptx.cuh"
#include "qmv_consumer.cuh"

namespace aq {

struct ChainRec {                // 128-byte aligned, as CUtensorMap is
    CUtensorMap tw, ts, tb;       // codes (128-byte swizzle), scales, biases
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    int M, N, K, tiles;           // tiles = ceil(N / 16)
    int flags;                    // AQ_CHAIN_INDEPENDENT
    int tile_base;                // tiles of the preceding matmuls since the last dependent one
    int pad[6];
};
static_assert(sizeof(ChainRec) % 128 == 0, "records must stay 128-byte aligned");

namespace {

using namespace dev;
using namespace qmv;

constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kMaxXBytes = 32768;
constexpr int kRedBytes = 2 * kConsumerWarps * kRows * 8 * 4;
constexpr int kNumBars = 2 * kStages + 4;                  // full[S], empty[S], red_full[2], red_empty[2]

struct ChainLayout {
    int x_off, xsum_off, red_off, bar_off, total;
};
__host__ __device__ inline ChainLayout chain_layout(int x_bytes) {
    ChainLayout L;
    L.x_off = kStages * kStageBytes;
    L.xsum_off = L.x_off + x_bytes;
    L.red_off = (L.xsum_off + x_bytes / 32 + 15) & ~15;  // M*K/64 floats = x_bytes/32 bytes
    L.bar_off = L.red_off + kRedBytes;
    L.total = L.bar_off + kNumBars * 8 + 16;   // + abort flag and the CTA-wide "go" word
    return L;
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ldg_cg_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

template <bool ONE_ROW>
__global__ void __launch_bounds__(kThreads, 2)
qmv_chain_kernel(const ChainRec *__restrict__ recs, int count, int *done, int x_bytes,
                 unsigned long long timeout_ns, int *status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t s_base = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (s_base - raw_base);
    const ChainLayout L = chain_layout(x_bytes);
    const uint32_t x_s = s_base + L.x_off;
    float *xsum = reinterpret_cast<float *>(smem + L.xsum_off);
    float *red = reinterpret_cast<float *>(smem + L.red_off);
    const uint32_t bar_full = s_base + L.bar_off;
    const uint32_t bar_empty = bar_full + kStages * 8;
    const uint32_t bar_red_full = bar_empty + kStages * 8;
    const uint32_t bar_red_empty = bar_red_full + 16;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bar_off + kNumBars * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(bar_red_full + 8 * p, kConsumerWarps);
            mbar_init(bar_red_empty + 8 * p, 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    auto set_abort = [&]() {
        if (!*abort_flag) {
            atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
            *abort_flag = 1;
        }
    };

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        int issued = 0;
        bool ok = true;
        for (int jm = 0; jm < count && ok; ++jm) {
            const ChainRec *rec = recs + jm;
            const int K = rec->K, T = rec->tiles;
            const int nblk = K / kBlockCodes;
            const int KB = (K + kStageCodes - 1) / kStageCodes;
            // tiles are dealt round-robin, continuing from the previous matmul
            // of the same dependency group so that the group stays balanced
            const int first = ((int)blockIdx.x - rec->tile_base % (int)gridDim.x + (int)gridDim.x) % (int)gridDim.x;
            for (int tile = first; tile < T && ok; tile += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb) {
                    const int slot = issued % kStages;
                    if (issued >= kStages &&
                        !mbar_wait_for(bar_empty + 8 * slot, ((issued / kStages) - 1) & 1, timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = s_base + slot * kStageBytes;
                    const uint32_t fb = bar_full + 8 * slot;
                    int nvalid = nblk - kb * kConsumerWarps;
                    nvalid = nvalid < kConsumerWarps ? nvalid : kConsumerWarps;
                    mbar_expect_tx(fb, (uint32_t)(nvalid * kCodeBlockBytes + 2 * kSBBytes));
                    for (int b = 0; b < nvalid; ++b)
                        tma_load_2d(dst + b * kCodeBlockBytes, &rec->tw, (kb * kConsumerWarps + b) * 32, tile * kRows,
                                    fb, pol);
                    tma_load_2d(dst + kCodesBytes, &rec->ts, kb * kStageGroups, tile * kRows, fb, pol);
                    tma_load_2d(dst + kCodesBytes + kSBBytes, &rec->tb, kb * kStageGroups, tile * kRows, fb, pol);
                    ++issued;
                }
            }
        }
        if (!ok) {
            set_abort();
            const uint64_t drain = global_timer() + timeout_ns;
            for (int it = (issued > kStages ? issued - kStages : 0); it < issued; ++it)
                while (!mbar_try_wait(bar_full + 8 * (it % kStages), (it / kStages) & 1) && global_timer() < drain) {
                }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // All eight consumer warps run every step below (named barriers need all
    // of them); after an abort the waits return at once and work is skipped.
    const int gid = lane >> 2;
    const int j = lane & 3;
    const int r0 = gid, r1 = gid + 8;
    const uint32_t xsum_s = smem_addr(xsum);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int par = 0, tcount = 0, item = 0;
    int prev_tiles_mine = 0, prev_tiles_total = 0;
    bool ok = true;

    volatile int *go = abort_flag + 1;  // CTA-wide decision, written by thread 0 between two barriers
    const __nv_bfloat16 *prev_x = nullptr;
    int prev_M = 0, prev_K = 0;
    for (int jm = 0; jm < count; ++jm) {
        const ChainRec *rec = recs + jm;
        const int M = rec->M, N = rec->N, K = rec->K, T = rec->tiles;
        const __nv_bfloat16 *x = rec->x;
        __nv_bfloat16 *y = rec->y;
        const int nblk = K / kBlockCodes;
        const int KB = (K + kStageCodes - 1) / kStageCodes;
        // A matmul flagged independent does not read the previous one's
        // output: it neither waits for it nor, when its x is the same buffer,
        // reloads x.  These decisions depend only on the plan, so every warp
        // passes the same sequence of named barriers.
        const bool dep = jm > 0 && !(rec->flags & AQ_CHAIN_INDEPENDENT);
        const bool new_x = jm == 0 || x != prev_x || M != prev_M || K != prev_K;
        if (jm > 0 && (dep || new_x)) {
            consumer_sync();  // every warp is done with the previous matmuls (tiles, y stores, x reads)
            if (threadIdx.x == 0) {
                if (dep && !*abort_flag) {
                    // every CTA has stored all its tiles of matmul jm-1
                    __threadfence();
                    atomicAdd(done + (jm - 1), prev_tiles_mine);
                    const uint64_t dl = global_timer() + timeout_ns;
                    while (ld_acquire_gpu(done + (jm - 1)) < prev_tiles_total) {
                        if (*abort_flag || global_timer() > dl) {
                            set_abort();
                            break;
                        }
                    }
                }
                *go = *abort_flag ? 0 : 1;
            }
            consumer_sync();
            if (!*go) {
                ok = false;
                break;
            }
        }
        prev_x = x;
        prev_M = M;
        prev_K = K;

        // ---- x of this matmul: L2 loads, word permutation, per-group sums
        if (new_x) {
            const int words = M * K / 8;
            for (int base = 0; base < words; base += 256) {
                const int wi = base + threadIdx.x;
                float part = 0.f;
                if (wi < words) {
                    const uint4 v = ldg_cg_v4(x + (size_t)wi * 8);
                    part = ((bf16lo(v.x) + bf16hi(v.x)) + (bf16lo(v.y) + bf16hi(v.y))) +
                           ((bf16lo(v.z) + bf16hi(v.z)) + (bf16lo(v.w) + bf16hi(v.w)));
                    uint4 p;
                    p.x = __byte_perm(v.x, v.z, 0x5410);
                    p.y = __byte_perm(v.x, v.z, 0x7632);
                    p.z = __byte_perm(v.y, v.w, 0x5410);
                    p.w = __byte_perm(v.y, v.w, 0x7632);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(x_s + wi * 16), "r"(p.x),
                                 "r"(p.y), "r"(p.z), "r"(p.w)
                                 : "memory");
                }
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 2);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 4);
                if (wi < words && (wi & 7) == 0) xsum[wi >> 3] = part;
            }
            consumer_sync();
        }

        ConsumerThread ct;
        consumer_init(ct, warp, lane, x_s, xsum_s, M, K);
        int mine = 0;

        const int first = ((int)blockIdx.x - rec->tile_base % (int)gridDim.x + (int)gridDim.x) % (int)gridDim.x;
        for (int tile = first; tile < T && ok; tile += gridDim.x) {  // on failure: abort, then barrier A
            ++mine;
            for (int kb = 0; kb < KB; ++kb, ++item) {
                const int slot = item % kStages;
                const uint32_t phase = (uint32_t)(item / kStages) & 1u;
                if (!mbar_wait_for(bar_full + 8 * slot, phase, timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const int blk = kb * kConsumerWarps + warp;
                if (blk < nblk) consume_shared_stage<ONE_ROW>(s_base + (uint32_t)(slot * kStageBytes), warp, lane, kb, ct, acc);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
            }
            if (!ok) break;
            // ---- tile finished: rotating reducer adds the eight partials in order
            const uint32_t rf = bar_red_full + 8 * par, re = bar_red_empty + 8 * par;
            float *rb = red + par * (kConsumerWarps * kRows * 8);
            if (tcount >= 2 && !mbar_wait_for(re, ((tcount >> 1) - 1) & 1, timeout_ns, abort_flag)) {
                ok = false;
                break;
            }
            float *rw = rb + warp * (kRows * 8);
            rw[r0 * 8 + 2 * j] = acc[0];
            rw[r0 * 8 + 2 * j + 1] = acc[1];
            rw[r1 * 8 + 2 * j] = acc[2];
            rw[r1 * 8 + 2 * j + 1] = acc[3];
            __syncwarp();
            if (lane == 0) mbar_arrive(rf);
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            if (warp == (tcount & (kConsumerWarps - 1))) {
                if (!mbar_wait_for(rf, (tcount >> 1) & 1, timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                for (int idx = lane; idx < kRows * M; idx += 32) {
                    const int m = idx / kRows, row = idx % kRows;
                    const int n = tile * kRows + row;
                    if (n < N) {
                        float v = rb[row * 8 + m];
#pragma unroll
                        for (int w = 1; w < kConsumerWarps; ++w) v += rb[w * (kRows * 8) + row * 8 + m];
                        y[(int64_t)m * N + n] = __float2bfloat16_rn(v);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(re);
            }
            ++tcount;
            par ^= 1;
        }
        if (!ok) {
            set_abort();   // the next barrier pair turns this into a CTA-wide stop
            ok = true;     // keep walking to barrier A with the other warps
        }
        prev_tiles_mine = mine;
        prev_tiles_total = T;
    }
    // the last matmul's counter, for completeness (nothing waits on it)
    consumer_sync();
    if (threadIdx.x == 0 && count > 0 && !*abort_flag) {
        __threadfence();
        atomicAdd(done + (count - 1), prev_tiles_mine);
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int kMaxDevices = 64;
std::atomic<int> g_attr_done[2][kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_smem_per_sm[kMaxDevices];

size_t records_bytes(int count) { return (size_t)count * sizeof(ChainRec); }
size_t counters_bytes(int count) { return ((size_t)count * sizeof(int) + 127) & ~(size_t)127; }

}  // namespace

size_t chain_workspace_bytes(int count) {
    if (count <= 0) return 0;
    return records_bytes(count) + counters_bytes(count);
}

namespace {

// Validates the descriptors (host only, no CUDA call).
aq_status chain_validate(const aq_matmul_desc *descs, int count, int group_size, int bits) {
    if (bits != 4 || group_size != 64) return AQ_ERR_UNSUPPORTED;
    for (int i = 0; i < count; ++i) {
        const aq_matmul_desc &d = descs[i];
        if (d.M < 1 || d.N < 1 || d.K < 1 || d.K % 64) return AQ_ERR_INVALID_ARG;
        if (d.flags & ~(int64_t)AQ_CHAIN_INDEPENDENT) return AQ_ERR_INVALID_ARG;
        if (!d.x || !d.w_packed || !d.scales || !d.biases || !d.y) return AQ_ERR_INVALID_ARG;
        if (d.M > 8 || d.K % 512 || d.M * d.K * 2 > kMaxXBytes || d.N > (int64_t)1 << 30) return AQ_ERR_UNSUPPORTED;
        if (!aligned(d.x, 16) || !aligned(d.w_packed, 16) || !aligned(d.scales, 16) || !aligned(d.biases, 16) ||
            !aligned(d.y, 2))
            return AQ_ERR_ALIGNMENT;
    }
    return AQ_OK;
}

// Encodes validated descriptors into host records and fills the plan's sizes.
aq_status chain_encode(const aq_matmul_desc *descs, int count, ChainRec *recs, aq_chain_plan *plan) {
    if (!encode_fn()) return AQ_ERR_UNSUPPORTED;
    int x_bytes = 16;
    bool one_row = true;
    for (int i = 0; i < count; ++i) {
        const aq_matmul_desc &d = descs[i];
        ChainRec &r = recs[i];
        std::memset(&r, 0, sizeof r);
        const uint64_t K = (uint64_t)d.K, N = (uint64_t)d.N, G = K / 64;
        if (!encode_2d(&r.tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, d.w_packed, K / 8, N, K / 2, 32, kRows,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&r.ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, d.scales, G, N, G * 2, kStageGroups, kRows,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_2d(&r.tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, d.biases, G, N, G * 2, kStageGroups, kRows,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
            return AQ_ERR_INVALID_ARG;
        r.x = static_cast<const __nv_bfloat16 *>(d.x);
        r.y = static_cast<__nv_bfloat16 *>(d.y);
        r.M = (int)d.M;
        r.N = (int)d.N;
        r.K = (int)d.K;
        r.tiles = (int)((d.N + kRows - 1) / kRows);
        r.flags = (int)d.flags;
        r.tile_base = (i > 0 && (d.flags & AQ_CHAIN_INDEPENDENT)) ? recs[i - 1].tile_base + recs[i - 1].tiles : 0;
        x_bytes = std::max(x_bytes, (int)(d.M * d.K * 2));
        one_row = one_row && d.M == 1;
    }
    plan->count = count;
    plan->x_bytes = (x_bytes + 15) & ~15;
    plan->one_row = one_row ? 1 : 0;
    return AQ_OK;
}

}  // namespace

aq_status chain_prepare(const aq_matmul_desc *descs, int count, int group_size, int bits, void *workspace,
                        size_t workspace_bytes, aq_chain_plan *plan, cudaError_t *err) {
    *err = cudaSuccess;
    if (!plan || count < 0) return AQ_ERR_INVALID_ARG;
    std::memset(plan, 0, sizeof *plan);
    if (count == 0) return AQ_OK;
    if (!descs || !workspace) return AQ_ERR_INVALID_ARG;
    if (bits != 4 || group_size != 64) return AQ_ERR_UNSUPPORTED;
    if (workspace_bytes < chain_workspace_bytes(count)) return AQ_ERR_INVALID_ARG;
    if (!aligned(workspace, 128)) return AQ_ERR_ALIGNMENT;
    aq_status st = chain_validate(descs, count, group_size, bits);  // before any CUDA call
    if (st != AQ_OK) return st;
    std::vector<ChainRec> recs((size_t)count);
    st = chain_encode(descs, count, recs.data(), plan);
    if (st != AQ_OK) return st;
    *err = cudaMemcpy(workspace, recs.data(), records_bytes(count), cudaMemcpyHostToDevice);
    if (*err != cudaSuccess) {
        std::memset(plan, 0, sizeof *plan);
        return AQ_ERR_CUDA;
    }
    plan->workspace = workspace;
    return AQ_OK;
}

cudaError_t chain_run(const aq_chain_plan *plan, uint64_t timeout_ns, int *status, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int sms = g_sms[dev].load(std::memory_order_relaxed);
    if (!sms) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sms[dev].store(sms, std::memory_order_relaxed);
    }
    int smem_sm = g_smem_per_sm[dev].load(std::memory_order_relaxed);
    if (!smem_sm) {
        e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e != cudaSuccess) return e;
        g_smem_per_sm[dev].store(smem_sm, std::memory_order_relaxed);
    }
    const int count = plan->count;
    const ChainLayout L = chain_layout(plan->x_bytes);
    const int smem = L.total + 1024;
    const bool one = plan->one_row != 0;
    auto kern = one ? qmv_chain_kernel<true> : qmv_chain_kernel<false>;
    if (!g_attr_done[one][dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 chain_layout(kMaxXBytes).total + 1024);
        if (e != cudaSuccess) return e;
        g_attr_done[one][dev].store(1, std::memory_order_release);
    }
    const int per_sm = std::max(1, std::min(2, smem_sm / (smem + 1024)));
    int *done = reinterpret_cast<int *>(static_cast<uint8_t *>(plan->workspace) + records_bytes(count));
    e = cudaMemsetAsync(done, 0, (size_t)count * sizeof(int), stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms * per_sm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const ChainRec *>(plan->workspace), count, done, plan->x_bytes,
                              (unsigned long long)timeout_ns, status);
}

// ---------------------------------------------------------------- allocation-free variant
//
// aq_chain_run_static runs the same kernel with its plan records and
// completion counters in the file-scope array below instead of a
// caller-provided workspace, for callers that cannot hand the library any
// device memory.  The array is fixed at kStaticChainMax matmuls (132 KB) and
// is held by every GPU that loads the library until the process exits.  Its
// device address is looked up once per device with cudaGetSymbolAddress (in
// host code the array's name is only a host-side stand-in).  Every call shares
// the array: calls that overlap on the GPU race, and the counters are cleared
// by every call before its launch.

constexpr int kStaticChainMax = 256;
static __device__ __align__(256) uint8_t g_static_chain_scratch[kStaticChainMax * sizeof(ChainRec) + 1024];

namespace {
std::atomic<void *> g_static_scratch_ptr[kMaxDevices];
std::mutex g_static_host_mutex;
ChainRec g_static_host_recs[kStaticChainMax];  // host staging of the records (no heap allocation)
}  // namespace

int chain_static_max() { return kStaticChainMax; }

aq_status chain_run_static(const aq_matmul_desc *descs, int count, int group_size, int bits, uint64_t timeout_ns,
                           int *status, cudaStream_t stream, cudaError_t *err) {
    *err = cudaSuccess;
    if (count < 0) return AQ_ERR_INVALID_ARG;
    if (count == 0) return AQ_OK;
    if (count > kStaticChainMax) return AQ_ERR_INVALID_ARG;  // beyond the static scratch
    if (!descs) return AQ_ERR_INVALID_ARG;
    aq_status st = chain_validate(descs, count, group_size, bits);  // before any CUDA call
    if (st != AQ_OK) return st;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return AQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return AQ_ERR_CUDA;
    }
    // set-up, once per device, with that device current
    void *scratch = g_static_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!scratch) {
        *err = cudaGetSymbolAddress(&scratch, g_static_chain_scratch);
        if (*err != cudaSuccess) return AQ_ERR_CUDA;
        g_static_scratch_ptr[dev].store(scratch, std::memory_order_release);
    }
    aq_chain_plan plan;
    std::memset(&plan, 0, sizeof plan);
    {
        std::lock_guard<std::mutex> lock(g_static_host_mutex);
        st = chain_encode(descs, count, g_static_host_recs, &plan);
        if (st != AQ_OK) return st;
        // from pageable memory: returns once the records are staged, so the
        // host buffer may be reused by the next call
        *err = cudaMemcpyAsync(scratch, g_static_host_recs, records_bytes(count), cudaMemcpyHostToDevice, stream);
        if (*err != cudaSuccess) return AQ_ERR_CUDA;
    }
    plan.workspace = scratch;
    *err = chain_run(&plan, timeout_ns, status, stream);  // clears the counters, then launches
    return *err == cudaSuccess ? AQ_OK : AQ_ERR_CUDA;
}

}  // namespace aq
