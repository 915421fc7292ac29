// Weight-streaming kernel for y = x . dequant(W)^T with 1..8 rows of x,
// fed by the Tensor Memory Accelerator.
//
// Decode time is the time to stream the packed weights ("epic: CUDA (MLX
// backend) prefill and decode acceleration program", Diagnosis; "gemma-4
// decode carries ~44 ms/token ...", re-scope paragraph).  This kernel keeps
// the weight stream going independently of the arithmetic:
//
//  * CTAs are persistent (two per SM); each walks its 16-row tiles of W
//    across the whole K in stages of 2048 codes, and each of its eight warps
//    owns one 256-code column block of every stage;
//  * every warp runs its own ring of shared-memory slots: it issues the TMA
//    copy of its next blocks' codes (cp.async.bulk.tensor, 128-byte swizzle)
//    and cp.async copies of the matching scales and biases, waits on its own
//    mbarrier, computes, and refills the slot it just consumed.  No warp waits
//    for another one to release a slot, so a slow warp never stalls the
//    others' weight stream;
//  * the arithmetic is the dequantization-free folded form (see
//    qmv_consumer.cuh): mma.sync m16n8k16 on exact bf16 codes 128 + q, one
//    LOP3 per code pair, fp32 fold per group of 64;
//  * at the end of a tile the eight warps' partial sums are added in a fixed
//    order by one rotating warp (mbarrier-guarded double buffer), so every
//    output is written exactly once and results are deterministic.
//
// Every wait is bounded by a global-timer deadline; on expiry the thread
// records AQ_ERR_TIMEOUT in the library's device status word, the CTA stops,
// and each warp first waits (also bounded) for the copies it issued.
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

constexpr int kThreads = kConsumerWarps * 32;
constexpr int kSlots = 4;                                  // ring slots per warp
constexpr int kSlotSBBytes = kRows * 8 * 2;                // scales then biases: 16 rows x 4 groups x 2 B each
constexpr int kMaxXBytes = 32768;                          // M*K*2 limit for staging x once per CTA
constexpr int kRedBytes = 2 * kConsumerWarps * kRows * 8 * 4;  // double-buffered cross-warp sums
// full[warp][slot], x, red_full[2], red_empty[2]
constexpr int kNumBars = kConsumerWarps * kSlots + 1 + 4;
constexpr int kCodesRegion = kConsumerWarps * kSlots * kCodeBlockBytes;  // 64 KB
constexpr int kSBRegion = kConsumerWarps * kSlots * kSlotSBBytes;        // 8 KB
constexpr int kMaxSmem = kCodesRegion + kSBRegion + kMaxXBytes + kMaxXBytes / 32 + 16 + kRedBytes + kNumBars * 8 +
                         16 + 1024;

struct Layout {
    int x_off;       // bf16 x, permuted, M*K*2 bytes
    int xsum_off;    // float [M][G]
    int red_off;     // float [2][8][16][8]
    int bar_off;     // uint64 [kNumBars] + abort flag
    int total;       // bytes (excluding the 1024 alignment slack)
};
__host__ __device__ inline Layout make_layout(int M, int K) {
    Layout L;
    const int x_bytes = (M * K * 2 + 15) & ~15;
    L.x_off = kCodesRegion + kSBRegion;
    L.xsum_off = L.x_off + x_bytes;
    L.red_off = (L.xsum_off + M * (K / 64) * 4 + 15) & ~15;
    L.bar_off = L.red_off + kRedBytes;
    L.total = L.bar_off + kNumBars * 8 + 16;
    return L;
}

__device__ __forceinline__ void cp_async_8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// ONE_ROW: M == 1 (only column 0 of the MMA output is used).
template <bool ONE_ROW>
__global__ void __launch_bounds__(kThreads, 2)
qmv_tma_kernel(const __grid_constant__ CUtensorMap tm_w, const uint16_t *__restrict__ scales,
               const uint16_t *__restrict__ biases, const __nv_bfloat16 *__restrict__ x,
               __nv_bfloat16 *__restrict__ y, int M, int N, int K, unsigned long long timeout_ns, int *status,
               int skip_x) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t s_base = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (s_base - raw_base);
    const Layout L = make_layout(M, K);
    const uint32_t codes_s = s_base;
    const uint32_t sb_s = s_base + kCodesRegion;
    const uint32_t x_s = s_base + L.x_off;
    float *xsum = reinterpret_cast<float *>(smem + L.xsum_off);
    float *red = reinterpret_cast<float *>(smem + L.red_off);
    const uint32_t bar_full = s_base + L.bar_off;                 // [warp][slot]
    const uint32_t bar_x = bar_full + kConsumerWarps * kSlots * 8;
    const uint32_t bar_red_full = bar_x + 8;                      // 2 barriers: partial sums written
    const uint32_t bar_red_empty = bar_red_full + 16;             // 2 barriers: partial sums consumed
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bar_off + kNumBars * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = K >> 6;
    const int nblk = K / kBlockCodes;                       // column blocks in K
    const int KB = (K + kStageCodes - 1) / kStageCodes;     // stages per tile
    const int T = (N + kRows - 1) / kRows;
    const int my_tiles = blockIdx.x < T ? (T - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int L_items = my_tiles * KB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kConsumerWarps * kSlots; ++i) mbar_init(bar_full + 8 * i, 1 + 32);
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

    const uint64_t pol = policy_evict_first();
    const uint32_t my_full = bar_full + (uint32_t)(warp * kSlots) * 8;
    const uint32_t my_codes = codes_s + (uint32_t)(warp * kSlots) * kCodeBlockBytes;
    const uint32_t my_sb = sb_s + (uint32_t)(warp * kSlots) * kSlotSBBytes;
    // this lane's scale (lanes 0-15) or bias (lanes 16-31) row of a block
    const int sb_row = lane & 15;
    const uint16_t *sb_src = (lane < 16 ? scales : biases);
    const uint32_t sb_dst_lane = (uint32_t)((lane >> 4) * (kRows * 8) + sb_row * 8);

    // Issue item `it` (tile, kb) into this warp's slot `slot`: one TMA box of
    // codes (lane 0) and one 8-byte cp.async of scales or biases per lane.
    auto issue = [&](int it, int slot) {
        const int tile = (int)blockIdx.x + (it / KB) * (int)gridDim.x;
        const int blk = (it % KB) * kConsumerWarps + warp;
        const uint32_t fb = my_full + 8 * slot;
        if (blk < nblk) {
            if (lane == 0) {
                mbar_expect_tx(fb, kCodeBlockBytes);
                tma_load_2d(my_codes + slot * kCodeBlockBytes, &tm_w, blk * 32, tile * kRows, fb, pol);
            }
            const int n = tile * kRows + sb_row;
            if (n < N) cp_async_8(my_sb + slot * kSlotSBBytes + sb_dst_lane, sb_src + (size_t)n * G + blk * 4);
        } else if (lane == 0) {
            mbar_arrive(fb);  // nothing to copy for this warp in the K tail
        }
        cp_async_arrive_noinc(fb);
    };

    // the weights do not depend on the preceding kernel: prefetch them first
    int issued = 0;
    for (; issued < kSlots && issued < L_items; ++issued) issue(issued, issued);
    griddep_wait();  // x comes from the preceding kernel; deadlines start after it
    if (threadIdx.x == 0 && !skip_x) {  // skip_x: test hook that leaves the x barrier incomplete
        mbar_expect_tx(bar_x, (uint32_t)(M * K * 2));
        for (int m = 0; m < M; ++m) bulk_load(x_s + m * K * 2, x + (int64_t)m * K, (uint32_t)(K * 2), bar_x);
    }

    bool ok = true;
    auto set_abort = [&]() {
        if (!*abort_flag) {
            atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
            *abort_flag = 1;
        }
    };
    if (!mbar_wait_for(bar_x, 0, timeout_ns, abort_flag)) ok = false;
    // permute each 8-element word of x to (x0,x4,x1,x5,x2,x6,x3,x7) and form
    // the per-group sums X[m,g] (8 lanes per group, fixed order)
    if (ok) {
        const int words = M * K / 8;
        for (int base = 0; base < words; base += kThreads) {
            const int wi = base + threadIdx.x;
            float part = 0.f;
            if (wi < words) {
                const uint32_t a = x_s + wi * 16;
                const uint4 v = lds128(a);
                part = ((bf16lo(v.x) + bf16hi(v.x)) + (bf16lo(v.y) + bf16hi(v.y))) +
                       ((bf16lo(v.z) + bf16hi(v.z)) + (bf16lo(v.w) + bf16hi(v.w)));
                uint4 pv;
                pv.x = __byte_perm(v.x, v.z, 0x5410);
                pv.y = __byte_perm(v.x, v.z, 0x7632);
                pv.z = __byte_perm(v.y, v.w, 0x5410);
                pv.w = __byte_perm(v.y, v.w, 0x7632);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pv.x), "r"(pv.y), "r"(pv.z),
                             "r"(pv.w)
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
    __syncthreads();

    ConsumerThread ct;
    consumer_init(ct, warp, lane, x_s, smem_addr(xsum), M, K);
    const int gid = lane >> 2, j = lane & 3;
    const int r0 = gid, r1 = gid + 8;
    const uint32_t sc_lane = (uint32_t)(gid * 8);   // scales of row r0 inside a slot; row r1 at +64, biases at +128

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int par = 0, tcount = 0;
    int kb = 0, tile = (int)blockIdx.x;
    int slot = 0;
    uint32_t phase = 0;
    for (int it = 0; ok && it < L_items; ++it) {
        if (!mbar_wait_for(my_full + 8 * slot, phase, timeout_ns, abort_flag)) {
            ok = false;
            break;
        }
        const int blk = kb * kConsumerWarps + warp;
        if (blk < nblk)
            consume_block<ONE_ROW, 64, kRows * 8>(my_codes + slot * kCodeBlockBytes,
                                                  my_sb + slot * kSlotSBBytes + sc_lane, kb, ct, acc);
        __syncwarp();
        if (issued < L_items) {
            fence_proxy_async();  // this warp's reads of the slot come before the copies that refill it
            issue(issued, slot);
            ++issued;
        }

        if (kb == KB - 1) {
            // Tile finished.  Every warp deposits its partial sums and moves
            // on; one warp per tile (rotating) adds the eight partials in a
            // fixed order and stores y.  Two buffers guarded by mbarriers.
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
            kb = 0;
            tile += (int)gridDim.x;
        } else {
            ++kb;
        }
        if (++slot == kSlots) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (!ok) {
        set_abort();
        // let this warp's copies in flight land before the CTA may exit: the
        // last kSlots items it issued (earlier ones were consumed)
        const uint64_t drain = global_timer() + timeout_ns;
        for (int k2 = (issued > kSlots ? issued - kSlots : 0); k2 < issued; ++k2)
            while (!mbar_try_wait(my_full + 8 * (k2 % kSlots), (uint32_t)(k2 / kSlots) & 1u) &&
                   global_timer() < drain) {
            }
        if (threadIdx.x == 0)
            while (!mbar_try_wait(bar_x, 0) && global_timer() < drain) {
            }
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
    CUtensorMap tw;
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.w, (uint64_t)K / 8, (uint64_t)N, (uint64_t)K / 2, 32, kRows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
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
    return cudaLaunchKernelEx(&cfg, kern, tw, a.scales, a.biases, static_cast<const __nv_bfloat16 *>(a.x),
                              static_cast<__nv_bfloat16 *>(a.y), M, N, K, (unsigned long long)a.timeout_ns,
                              a.status, a.debug_skip_x ? 1 : 0);
}

}  // namespace aq
