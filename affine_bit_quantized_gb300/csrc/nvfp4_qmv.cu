// Weight-streaming kernel for y = x . W^T with NVFP4 weights and 1..8 rows of x.
//
// The "MLX CUDA Cleanup Plan" page (Refactor Plan, Phase 3b) asks for a CUDA
// NVFP4 qmv for its mode=nvfp4, group_size=16 checkpoint, kept structurally
// separate from the affine path.  The format and the consumer arithmetic are
// in nvfp4_consumer.cuh (shared with the NVFP4 mode of the chain kernel); the
// stream and the tile bookkeeping are those of the affine decode kernel (a TMA
// producer warp filling a ring of 36 KB stages, sixteen consumer warps, a
// reducer warp adding their partials in a fixed order).  x is bulk-copied
// once per CTA and converted in place to scaled fp16 in the consumer's order,
// with one power-of-two scale per row (the partial sums are scaled back, then
// the reducer multiplies by the tensor scale before the one bf16 rounding).
//
// Every mbarrier wait is bounded (global-timer deadline, device status word),
// as in the affine kernels.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "aq_internal.h"
#include "aq_ptx.cuh"
#include "nvfp4_consumer.cuh"
#include "qmv_consumer.cuh"

namespace aq {
namespace {

using namespace dev;
using namespace qmv;

constexpr int kThreads = (kConsumerWarps + 2) * 32;   // consumers, TMA producer, reducer
constexpr int kNS = 4;                                 // ring depth (room for the bars)
constexpr int kCodes = kNvCodes;                       // codes per row and stage (1024 bytes)
constexpr int kStage = kNvStage;                       // 36864
constexpr int kNumBars = 2 * kNS + 1 + 8;              // full[4], empty[4], x, red_full[4], red_empty[4]
constexpr int kSmemLimit = 232448;

struct Layout {
    int x_off, xinfo_off, red_off, bar_off, total;
};
// ns: ring depth, 4 beside x of up to 32 KB, 3 beside x of up to 64 KB
__host__ __device__ inline Layout make_layout(int M, int K, int ns) {
    Layout L;
    L.x_off = ns * kStage;
    L.xinfo_off = L.x_off + M * x_row_bytes(M, K);
    L.red_off = L.xinfo_off + kXInfoBytes;
    L.bar_off = L.red_off + red_bytes(M);
    L.total = L.bar_off + kNumBars * 8 + 16;
    return L;
}

// x [M][K] bf16, bulk-copied to `raw` (rows x_row_bytes apart) -> fp16 in
// place, in the staged order of nvfp4_consumer.cuh, each row times 2^e (e from its max |x|, as in the
// affine staging), and inv_scale[m] = 2^-e.
template <bool ONE_ROW, int XROOM>
__device__ __forceinline__ void stage_x_fp16(uint32_t raw, uint32_t xinfo, int M_, int K) {
    const int M = ONE_ROW ? 1 : M_;
    const int tid = threadIdx.x;
    const int wpr = K / 8, words = M * wpr, xrb = x_row_bytes(M, K);
    int *row_max = reinterpret_cast<int *>(__cvta_shared_to_generic(xinfo));
    float *inv_scale = reinterpret_cast<float *>(__cvta_shared_to_generic(xinfo + 64));
    uint4 v[XROOM / 16 / kConsumerThreads];
#pragma unroll
    for (int u = 0; u < XROOM / 16 / kConsumerThreads; ++u) {
        if (u * kConsumerThreads >= words) break;   // uniform over the CTA
        const int wi = u * kConsumerThreads + tid;
        int mx = 0;
        if (wi < words) {
            const int m = ONE_ROW ? 0 : wi / wpr, wr = wi - m * wpr;
            v[u] = lds128(raw + (uint32_t)(m * xrb + wr * 16));
            mx = max(max(bf16x2_abs_max(v[u].x), bf16x2_abs_max(v[u].y)),
                     max(bf16x2_abs_max(v[u].z), bf16x2_abs_max(v[u].w)));
        }
        mx = __reduce_max_sync(0xFFFFFFFFu, mx);
        if ((tid & 31) == 0 && wi < words) atomicMax(row_max + (ONE_ROW ? 0 : wi / wpr), mx);
    }
    consumer_sync();
#pragma unroll
    for (int u = 0; u < XROOM / 16 / kConsumerThreads; ++u) {
        if (u * kConsumerThreads >= words) break;
        const int wi = u * kConsumerThreads + tid;
        if (wi < words) {
            const int m = ONE_ROW ? 0 : wi / wpr, wr = wi - m * wpr;
            const float sc = pow2f(x_scale_exponent(row_max[m]));
            const uint4 a = v[u];
            // into the consumer's order within the word's 128-code block (every
            // word of the block was read before the barrier above)
            const uint32_t q = raw + (uint32_t)(m * xrb + (wr >> 4) * 256) + nv_x_word_offset(wr & 15);
            sts64u(q, f32x2_to_f16x2(bf16lo(a.x) * sc, bf16hi(a.x) * sc), f32x2_to_f16x2(bf16lo(a.y) * sc, bf16hi(a.y) * sc));
            sts64u(q + 32, f32x2_to_f16x2(bf16lo(a.z) * sc, bf16hi(a.z) * sc),
                   f32x2_to_f16x2(bf16lo(a.w) * sc, bf16hi(a.w) * sc));
        }
    }
    if (tid < M) inv_scale[tid] = pow2f(-x_scale_exponent(row_max[tid]));
    consumer_sync();
}

// group: CTAs per group (1: each CTA takes all M rows).  With group G > 1, CTA
// g of each group takes rows [g rows, (g + 1) rows) of x and y, and the G CTAs
// walk the same tiles at the same pace, so that W mostly comes from DRAM once
// and from L2 for the others.
template <bool ONE_ROW, int NS>
__global__ void __launch_bounds__(kThreads, 1)
nvfp4_qmv_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                 const __nv_bfloat16 *__restrict__ x, __nv_bfloat16 *__restrict__ y, int M, int N, int K,
                 float global_scale, unsigned long long timeout_ns, int *status, int group, int rows) {
    // the CTA's place among those walking the tiles (a group counts once)
    const int cta = (int)blockIdx.x / group, ncta = (int)gridDim.x / group;
    if (group > 1) {
        const int m0 = ((int)blockIdx.x % group) * rows;
        x += (size_t)m0 * K;
        y += (size_t)m0 * N;
        M = M - m0 < rows ? M - m0 : rows;
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Layout L = make_layout(M, K, NS);
    const uint32_t s_base = smem_addr(smem);
    const uint32_t x_s = s_base + (uint32_t)L.x_off;
    const uint32_t xinfo = s_base + (uint32_t)L.xinfo_off;
    const float *inv_scale = reinterpret_cast<const float *>(smem + L.xinfo_off + 64);
    const uint32_t bar_full = s_base + L.bar_off;
    const uint32_t bar_empty = bar_full + kNS * 8;
    const uint32_t bar_x = bar_empty + kNS * 8;
    const uint32_t bar_red = bar_x + 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bar_off + kNumBars * 8);
    TileCtx tc;
    tc.red = reinterpret_cast<float *>(smem + L.red_off);
    tc.red_full = bar_red;
    tc.red_empty = bar_red + 32;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = (K + kCodes - 1) / kCodes;   // stages per tile
    const int T = (N + kRows - 1) / kRows;
    const int my_tiles = cta < T ? (T - 1 - cta) / ncta + 1 : 0;
    const int items = my_tiles * KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_x, 1);
        for (int p = 0; p < red_bufs<ONE_ROW>(); ++p) {
            mbar_init(tc.red_full + 8 * p, kConsumerWarps);
            mbar_init(tc.red_empty + 8 * p, 1);
        }
        for (int m = 0; m < 2 * kMaxM; ++m) reinterpret_cast<int *>(smem + L.xinfo_off)[m] = 0;
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    griddep_launch();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            auto issue = [&](int it) {
                const int slot = it % NS, tile = cta + (it / KB) * ncta, kb = it % KB;
                const uint32_t dst = s_base + slot * kStage, fb = bar_full + 8 * slot;
                // codes: one box of 8 chunks x 32 rows x 128 bytes; scales: 128 bytes x 32 rows
                // (parts past the row's end read as zeros and still count)
                mbar_expect_tx(fb, (uint32_t)kStage);
                tma_load_3d(dst, &tm_w, 0, tile * kRows, kb * kBoxes, fb, pol);
                tma_load_2d(dst + kCodesBytes, &tm_s, kb * (kCodes / 16), tile * kRows, fb, pol);
            };
            int issued = 0;
            bool ok = true;
            for (; issued < items && issued < NS; ++issued) issue(issued);   // weights first
            griddep_wait();
            const uint64_t deadline = global_timer() + timeout_ns;
            mbar_expect_tx(bar_x, (uint32_t)(M * K * 2));
            for (int m = 0; m < M; ++m)
                bulk_load(x_s + m * x_row_bytes(M, K), x + (int64_t)m * K, (uint32_t)(K * 2), bar_x);
            for (; issued < items; ++issued) {
                const int slot = issued % NS;
                if (!mbar_wait(bar_empty + 8 * slot, ((issued / NS) - 1) & 1, deadline, abort_flag)) {
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
                const uint64_t drain = global_timer() + timeout_ns;
                for (int it = (issued > NS ? issued - NS : 0); it < issued; ++it)
                    while (!mbar_try_wait(bar_full + 8 * (it % NS), (it / NS) & 1) && global_timer() < drain) {
                    }
                while (!mbar_try_wait(bar_x, 0) && global_timer() < drain) {
                }
            }
        }
        __syncwarp();
    } else if (warp == kConsumerWarps + 1) {
        // ------------------------------------------------------------ reducer
        bool ok = true;
        for (int t = 0; ok && t < my_tiles; ++t)
            ok = reduce_tile<ONE_ROW>(tc, t, cta + t * ncta, M, N, y, lane, timeout_ns,
                                      abort_flag, nullptr, 0, 1, global_scale);
        if (!ok && lane == 0 && !*abort_flag) {
            atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------------ consumers
        griddep_wait();
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
        stage_x_fp16<ONE_ROW, NS == kNS ? kMaxXBytes : 2 * kMaxXBytes>(x_s, xinfo, M, K);
        const int gid = lane >> 2, t = lane & 3;
        NvThread ct;
        nv_consumer_init(ct, warp, lane);
        const int M1 = ONE_ROW ? 1 : M;
        const int xrow = ONE_ROW ? 0 : (gid < M1 ? gid : M1 - 1);    // B column gid holds x row gid
        const uint32_t xq0 = x_s + (uint32_t)(xrow * x_row_bytes(M1, K) + warp * 256 + t * 8);
        const int nblk = K / 128;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        // the row scales of this lane's MMA columns 2t and 2t + 1
        const float inv[2] = {inv_scale[2 * t < M1 ? 2 * t : M1 - 1], inv_scale[2 * t + 1 < M1 ? 2 * t + 1 : M1 - 1]};
        bool ok = alive && !*abort_flag;
        int item = 0;
        for (int tl = 0; tl < my_tiles; ++tl) {
            for (int kb = 0; ok && kb < KB; ++kb, ++item) {
                const int slot = item % NS;
                if (!mbar_wait_fast(bar_full + 8 * slot, (uint32_t)(item / NS) & 1u, deadline, abort_flag)) {
                    ok = false;
                    break;
                }
                if (kb * kConsumerWarps + warp < nblk)
                    consume_stage_nvfp4(s_base + (uint32_t)(slot * kStage), ct, xq0 + (uint32_t)(kb * kCodes * 2), acc);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
            }
            if (ok) ok = deposit_tile<ONE_ROW>(tc, acc, tl, M, warp, lane, lane >> 2, inv, timeout_ns, abort_flag);
        }
        if (!ok) fail();
    }
}

bool encode_scales_2d(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)(kCodes / 16), (cuuint32_t)kRows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_attr_done[4][kMaxDevices];

}  // namespace

cudaError_t launch_nvfp4_qmv(const Nvfp4Args &a) {
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
    // M: rows of x per CTA; G CTAs per group of CTAs walking the same tiles
    const int M = a.rows > 0 && a.rows < a.M ? a.rows : (int)a.M, N = (int)a.N, K = (int)a.K;
    const int G = (int)((a.M + M - 1) / M);
    if (G > sms) return cudaErrorInvalidConfiguration;
    const bool one = M == 1;
    // x beyond 32 KB (up to 64 KB): a 3-stage ring beside it
    const bool ns3 = (int64_t)M * K * 2 > kMaxXBytes;
    auto kern = ns3 ? (one ? nvfp4_qmv_kernel<true, 3> : nvfp4_qmv_kernel<false, 3>)
                    : (one ? nvfp4_qmv_kernel<true, kNS> : nvfp4_qmv_kernel<false, kNS>);
    const int ki = 2 * (int)ns3 + (int)one;
    if (!g_attr_done[ki][dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        g_attr_done[ki][dev].store(1, std::memory_order_release);
    }
    const Layout L = make_layout(M, K, ns3 ? 3 : kNS);
    const int smem = L.total + 1024;
    if (smem > kSmemLimit) return cudaErrorInvalidConfiguration;
    CUtensorMap tw, ts;
    if (!tensor_map_encoder() || !encode_codes_3d(&tw, a.w, (uint64_t)K / 2, (uint64_t)N) ||
        !encode_scales_2d(&ts, a.scales, (uint64_t)K / 16, (uint64_t)N))
        return cudaErrorInvalidValue;
    const int T = (N + kRows - 1) / kRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(G * std::min(T, sms / G)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tw, ts, static_cast<const __nv_bfloat16 *>(a.x),
                              static_cast<__nv_bfloat16 *>(a.y), (int)a.M, N, K, a.global_scale,
                              (unsigned long long)a.timeout_ns, a.status, G, M);
}

}  // namespace aq
