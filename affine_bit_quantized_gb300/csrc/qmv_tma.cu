// Weight-streaming kernel for y = x . dequant(W)^T with 1..8 rows of x,
// fed by the Tensor Memory Accelerator.
//
// Decode time is the time to stream the packed weights ("epic: CUDA (MLX
// backend) prefill and decode acceleration program", Diagnosis; "gemma-4
// decode carries ~44 ms/token ...", re-scope paragraph).  This kernel keeps
// the weight stream going independently of the arithmetic:
//
//  * one producer warp per CTA copies 16-row x 2048-code tiles of the packed
//    codes, plus the matching scales and biases, into a ring of shared-memory
//    stages with cp.async.bulk.tensor (TMA), completion tracked by mbarriers;
//  * eight consumer warps each take one 256-code column block of a stage
//    (16 rows x 4 groups) and run the dequantization-free dot product of
//    the folded form on mma.sync m16n8k16 (bf16 in, fp32 out):
//        D[n,m,g] = sum_{k in g} (128 + q[n,k]) * x[m,k]
//        y[m,n]  += scale[n,g] * D[n,m,g] + (bias[n,g] - 128*scale[n,g]) * X[m,g]
//    with X[m,g] = sum_{k in g} x[m,k] computed once per CTA;
//  * CTAs are persistent: each walks its 16-row tiles across the whole K,
//    the eight warps' partial sums are combined in shared memory in a fixed
//    order, and every output is written exactly once (deterministic).
//
// A code q is turned into the exact bf16 value 128 + q by OR-ing its nibble
// into the mantissa of 128.0: one LOP3 makes the pair (q[p], q[p+4]) of a
// word; x is stored in shared memory with each 8-element word permuted to
// (x0,x4,x1,x5,x2,x6,x3,x7) so that the MMA's B fragment matches those pairs
// (a dot product is indifferent to the order of k).
//
// The code tiles use the TMA 128-byte swizzle, so the consumers' 8-byte
// shared-memory reads of 8 rows at once are free of bank conflicts.
//
// Every mbarrier wait is bounded by a global-timer deadline; on expiry the
// thread records AQ_ERR_TIMEOUT in the library's device status word, the CTA
// stops, and the producer first waits (also bounded) for the copies it
// issued.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "aq_internal.h"
#include "aq_ptx.cuh"
#include "qmv_consumer.cuh"

namespace aq {
namespace {

using namespace dev;
using namespace qmv;

constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kMaxXBytes = 32768;                          // M*K*2 limit for staging x once per CTA
constexpr int kRedBytes = 2 * kConsumerWarps * kRows * 8 * 4;  // double-buffered cross-warp sums
// largest layout: x of 32 KB, X sums of M*K/16 bytes, barriers, alignment slack
constexpr int kNumBars = 2 * kStages + 1 + 4;   // full[S], empty[S], x, red_full[2], red_empty[2]
constexpr int kMaxSmem = kStages * kStageBytes + kMaxXBytes + kMaxXBytes / 16 + 16 + kRedBytes + kNumBars * 8 +
                         16 + 1024;

struct Layout {
    int x_bytes;     // M*K*2 rounded up to 16
    int xsum_off;    // float [M][G]
    int red_off;     // float [2][8][16][8]
    int bar_off;     // uint64 [kNumBars] + abort flag
    int total;       // bytes (excluding the 1024 alignment slack)
};
__host__ __device__ inline Layout make_layout(int M, int K) {
    Layout L;
    L.x_bytes = (M * K * 2 + 15) & ~15;
    const int x_off = kStages * kStageBytes;
    L.xsum_off = x_off + L.x_bytes;
    L.red_off = (L.xsum_off + M * (K / 64) * 4 + 15) & ~15;
    L.bar_off = L.red_off + kRedBytes;
    L.total = L.bar_off + kNumBars * 8 + 16;
    return L;
}

// ONE_ROW: M == 1 (only column 0 of the MMA output is used).
template <bool ONE_ROW>
__global__ void __launch_bounds__(kThreads, 2)
qmv_tma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
               const __grid_constant__ CUtensorMap tm_b, const __nv_bfloat16 *__restrict__ x,
               __nv_bfloat16 *__restrict__ y, int M, int N, int K, unsigned long long timeout_ns,
               int *status, int skip_x) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Layout L = make_layout(M, K);
    const uint32_t s_base = smem_addr(smem);
    const uint32_t x_s = s_base + kStages * kStageBytes;
    float *xsum = reinterpret_cast<float *>(smem + L.xsum_off);
    float *red = reinterpret_cast<float *>(smem + L.red_off);
    const uint32_t bar_full = s_base + L.bar_off;          // kStages barriers
    const uint32_t bar_empty = bar_full + kStages * 8;     // kStages barriers
    const uint32_t bar_x = bar_empty + kStages * 8;
    const uint32_t bar_red_full = bar_x + 8;               // 2 barriers: partial sums written
    const uint32_t bar_red_empty = bar_red_full + 16;      // 2 barriers: partial sums consumed
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bar_off + kNumBars * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nblk = K / kBlockCodes;                       // column blocks in K
    const int KB = (K + kStageCodes - 1) / kStageCodes;     // stages per tile
    const int T = (N + kRows - 1) / kRows;
    const int my_tiles = blockIdx.x < T ? (T - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int L_items = my_tiles * KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_x, 1);
        for (int p = 0; p < 2; ++p) {
            mbar_init(bar_red_full + 8 * p, kConsumerWarps);
            mbar_init(bar_red_empty + 8 * p, 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    griddep_launch();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        auto issue = [&](int it) {
            const int slot = it % kStages;
            const int tile = (int)blockIdx.x + (it / KB) * (int)gridDim.x;
            const int kb = it % KB;
            const uint32_t dst = s_base + slot * kStageBytes;
            const uint32_t fb = bar_full + 8 * slot;
            int nvalid = nblk - kb * kConsumerWarps;
            nvalid = nvalid < kConsumerWarps ? nvalid : kConsumerWarps;
            mbar_expect_tx(fb, (uint32_t)(nvalid * kCodeBlockBytes + 2 * kSBBytes));
            for (int b = 0; b < nvalid; ++b)
                tma_load_2d(dst + b * kCodeBlockBytes, &tm_w, (kb * kConsumerWarps + b) * 32, tile * kRows, fb, pol);
            tma_load_2d(dst + kCodesBytes, &tm_s, kb * kStageGroups, tile * kRows, fb, pol);
            tma_load_2d(dst + kCodesBytes + kSBBytes, &tm_b, kb * kStageGroups, tile * kRows, fb, pol);
        };
        int issued = 0;
        bool ok = true;
        // the weights do not depend on the preceding kernel: prefetch them first
        for (; issued < L_items && issued < kStages; ++issued) issue(issued);
        griddep_wait();
        const uint64_t deadline = global_timer() + timeout_ns;
        if (!skip_x) {  // skip_x: test hook that leaves the x barrier incomplete
            mbar_expect_tx(bar_x, (uint32_t)(M * K * 2));
            for (int m = 0; m < M; ++m) bulk_load(x_s + m * K * 2, x + (int64_t)m * K, (uint32_t)(K * 2), bar_x);
        }
        for (; issued < L_items; ++issued) {
            const int slot = issued % kStages;
            if (!mbar_wait(bar_empty + 8 * slot, ((issued / kStages) - 1) & 1, deadline, abort_flag)) {
                ok = false;
                break;
            }
            issue(issued);
        }
        if (!ok) {
            if (!*abort_flag) {
                atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
                *abort_flag = 1;
            }
            // let the copies already issued land before the CTA can exit
            const uint64_t drain = global_timer() + timeout_ns;
            for (int it = (issued > kStages ? issued - kStages : 0); it < issued; ++it)
                while (!mbar_try_wait(bar_full + 8 * (it % kStages), (it / kStages) & 1) && global_timer() < drain) {
                }
            while (!mbar_try_wait(bar_x, 0) && global_timer() < drain) {
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Every consumer warp runs the whole loop, even after a timeout, because
    // the named barriers below need all of them; after an abort the waits
    // return at once and the work is skipped.
    const int gid = lane >> 2;
    const int j = lane & 3;
    const int r0 = gid, r1 = gid + 8;
    griddep_wait();  // x comes from the preceding kernel; the deadline starts after it
    const uint64_t deadline = global_timer() + timeout_ns;
    bool alive = true;
    auto fail = [&]() {
        if (alive && !*abort_flag) {
            atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
            *abort_flag = 1;
        }
        alive = false;
    };

    if (!mbar_wait(bar_x, 0, deadline, abort_flag)) fail();
    // permute each 8-element word of x to (x0,x4,x1,x5,x2,x6,x3,x7) and form
    // the per-group sums X[m,g] (8 lanes per group, fixed order)
    if (alive) {
        const int words = M * K / 8;
        for (int base = 0; base < words; base += 256) {
            const int wi = base + threadIdx.x;
            float part = 0.f;
            if (wi < words) {
                const uint32_t a = x_s + wi * 16;
                const uint4 v = lds128(a);
                part = ((bf16lo(v.x) + bf16hi(v.x)) + (bf16lo(v.y) + bf16hi(v.y))) +
                       ((bf16lo(v.z) + bf16hi(v.z)) + (bf16lo(v.w) + bf16hi(v.w)));
                uint4 p;
                p.x = __byte_perm(v.x, v.z, 0x5410);
                p.y = __byte_perm(v.x, v.z, 0x7632);
                p.z = __byte_perm(v.y, v.w, 0x5410);
                p.w = __byte_perm(v.y, v.w, 0x7632);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(p.x), "r"(p.y), "r"(p.z),
                             "r"(p.w)
                             : "memory");
            }
            part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);
            part += __shfl_xor_sync(0xFFFFFFFFu, part, 2);
            part += __shfl_xor_sync(0xFFFFFFFFu, part, 4);
            // word wi of the x buffer belongs to row m = wi / (K/8), group (wi mod K/8) / 8,
            // i.e. to X[m*G + g] with index wi / 8
            if (wi < words && (wi & 7) == 0) xsum[wi >> 3] = part;
        }
    }
    consumer_sync();

    ConsumerThread ct;
    consumer_init(ct, warp, lane, x_s, smem_addr(xsum), M, K);

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int par = 0, tcount = 0;
    int kb = 0, tile = (int)blockIdx.x;
    uint32_t phase = 0;
    bool ok = alive;
    for (int it0 = 0; ok && it0 < L_items; it0 += kStages, phase ^= 1u) {
#pragma unroll
        for (int slot = 0; slot < kStages; ++slot) {
            if (it0 + slot >= L_items) break;
            if (!mbar_wait_fast(bar_full + 8 * slot, phase, deadline, abort_flag)) {
                ok = false;
                break;
            }
            const int blk = kb * kConsumerWarps + warp;
            if (blk < nblk) consume_shared_stage<ONE_ROW>(s_base + (uint32_t)(slot * kStageBytes), warp, lane, kb, ct, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);

            if (kb == KB - 1) {
                // Tile finished.  Every warp deposits its partial sums and moves
                // on; one warp per tile (rotating) adds the eight partials in a
                // fixed order and stores y.  Two buffers guarded by mbarriers,
                // so no CTA-wide barrier stalls the pipeline.
                const uint32_t rf = bar_red_full + 8 * par, re = bar_red_empty + 8 * par;
                float *rb = red + par * (kConsumerWarps * kRows * 8);
                if (tcount >= 2 && !mbar_wait_fast(re, ((tcount >> 1) - 1) & 1, deadline, abort_flag)) {
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
                    if (!mbar_wait_fast(rf, (tcount >> 1) & 1, deadline, abort_flag)) {
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
                kb = 0;
                tile += (int)gridDim.x;
            } else {
                ++kb;
            }
        }
    }
    if (!ok) fail();
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

constexpr int kMaxDevices = 64;
constexpr int kMaxCtasPerSm = 2;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_smem_per_sm[kMaxDevices];
std::atomic<int> g_attr_done[2][kMaxDevices];

}  // namespace

bool qmv_tma_supported(const MatmulArgs &a) {
    return a.M >= 1 && a.M <= 8 && a.K % 512 == 0 && a.M * a.K * 2 <= kMaxXBytes && encode_fn() != nullptr &&
           (reinterpret_cast<uintptr_t>(a.scales) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.biases) & 15) == 0;
}

cudaError_t launch_qmv_tma(const MatmulArgs &a) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int sms = g_sms[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sms[dev].store(sms, std::memory_order_relaxed);
    }
    int smem_sm = g_smem_per_sm[dev].load(std::memory_order_relaxed);
    if (smem_sm == 0) {
        e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e != cudaSuccess) return e;
        g_smem_per_sm[dev].store(smem_sm, std::memory_order_relaxed);
    }
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K;
    const Layout L = make_layout(M, K);
    const int smem = L.total + 1024;
    const bool one = (M == 1);
    auto kern = one ? qmv_tma_kernel<true> : qmv_tma_kernel<false>;
    if (!g_attr_done[one][dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return e;
        g_attr_done[one][dev].store(1, std::memory_order_release);
    }
    CUtensorMap tw, ts, tb;
    const int G = K / 64;
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.w, (uint64_t)K / 8, (uint64_t)N, (uint64_t)K / 2, 32, kRows,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, (uint64_t)G, (uint64_t)N, (uint64_t)G * 2,
                   kStageGroups, kRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.biases, (uint64_t)G, (uint64_t)N, (uint64_t)G * 2,
                   kStageGroups, kRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const int T = (N + kRows - 1) / kRows;
    // CTAs per SM that fit in shared memory (1 KB per CTA is reserved by the
    // system).  Two CTAs per SM measured faster than one, also in a chain of
    // launches with programmatic dependent launch.
    const int per_sm = std::max(1, std::min(kMaxCtasPerSm, smem_sm / (smem + 1024)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(T, sms * per_sm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tw, ts, tb, static_cast<const __nv_bfloat16 *>(a.x),
                              static_cast<__nv_bfloat16 *>(a.y), M, N, K, (unsigned long long)a.timeout_ns,
                              a.status, a.debug_skip_x ? 1 : 0);
}

}  // namespace aq
