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
//    TMA kernel (qmv_tma.cu): 32-row x 2048-code stages through a 4-stage
//    shared-memory ring, mma.sync on exact fp16 codes 1024 + q, per-group fold
//    (qmv_consumer.cuh);
//  * the producer walks the matmuls in order and keeps streaming the NEXT
//    matmuls' weights while the consumers wait for a dependency, because
//    weights never depend on earlier outputs;
//  * matmul j reads its x only after every CTA has stored all of its tiles of
//    matmul j-1 (a completion counter per dependency group in the caller's
//    workspace, bounded wait), which is the same ordering a chain of
//    stream-ordered launches gives; the count is published with a GPU-scope
//    release, and polled with an acquire, where a later matmul reads or
//    rewrites memory written up to the group (or rewrites memory read up to
//    it), as the host finds when it encodes the plan;
//  * matmuls may hold 4- or 8-bit affine codes, or NVFP4 weights (one format
//    per chain).
//
// The plan (one record per matmul: three TMA descriptors plus pointers and
// sizes) and the counters live in caller-owned device memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstddef>
#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

#include "aq.h"
#include "aq_internal.h"
#include "aq_ptx.cuh"
#include "nvfp4_consumer.cuh"
#include "qmv_consumer.cuh"

namespace aq {

struct ChainRec {                // 128-byte aligned, as CUtensorMap is
    CUtensorMap tw, ts, tb;       // codes (128-byte swizzle), scales and biases (swizzled boxes);
                                  // NVFP4: E4M3 scales in ts (tb a copy of it)
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    int M, N, K, tiles;           // tiles = ceil(N / 32)
    int flags;                    // AQ_CHAIN_INDEPENDENT, and kRecRelease (set by the host)
    int tile_base;                // tiles of the preceding matmuls since the last dependent one
    int bits;                     // code width: 4 or 8
    int group;                    // first matmul of this one's dependency group (its counter)
    const float *gscale;          // NVFP4: the tensor's fp32 scale (device); else unused
    int pad[2];
};
static_assert(sizeof(ChainRec) % 128 == 0, "records must stay 128-byte aligned");

// Record flag set by the host on the last matmul of a dependency group whose
// completion must be published with a GPU-scope release (and acquired by the
// next group's poll): some later matmul of the chain reads or rewrites memory
// that a matmul up to this group wrote, or rewrites memory one of them read.
// Without it the group's completion counter is a relaxed atomic: the next
// group still starts only after every tile of this one is stored, but no
// memory fence waits for those stores to reach L2 (≈ 0.9 us per group).
constexpr int kRecRelease = 0x10000000;
static_assert(offsetof(ChainRec, x) % 16 == 0 && offsetof(ChainRec, M) == offsetof(ChainRec, x) + 16 &&
                  offsetof(ChainRec, flags) == offsetof(ChainRec, x) + 32 &&
                  offsetof(ChainRec, bits) == offsetof(ChainRec, x) + 40 &&
                  offsetof(ChainRec, group) == offsetof(ChainRec, x) + 44,
              "the scalar part of a record is read as three 16-byte vectors");

namespace {

using namespace dev;
using namespace qmv;

constexpr int kThreads = (kConsumerWarps + 2) * 32;   // consumers, TMA producer, reducer/signaller
constexpr int kMaxStages = 4;   // ring depth (36 KB stages); 5 measured no faster
constexpr int kNumBars = 2 * kMaxStages + 9;   // full[S], empty[S], red_full[4], red_empty[4], dep
constexpr int kSmemLimit = 232448;           // dynamic shared memory a CTA may use

constexpr int kInfoCap = 256;   // records whose scalar part is kept in shared memory (48 bytes each)

struct ChainLayout {
    int stages;  // ring depth (kMaxStages)
    int xq_off, wq, xsum_off, ws, red_off, info_off, bar_off, total;
};
// x_bytes: the largest staging room of the chain's x (x_stage_bytes: M * K * 2
// with K in whole stages); max_m: its largest M.  Each consumer warp has its
// own region of x fragments and of (Xs, X') sums.
__host__ __device__ inline ChainLayout chain_layout(int x_bytes, int max_m) {
    ChainLayout L;
    L.stages = kMaxStages;   // fits beside the largest rest (x of 32 KB, M = 8)
    L.xq_off = L.stages * kStageBytes;
    L.wq = xw_region_bytes(x_bytes, max_m);
    L.xsum_off = L.xq_off + kConsumerWarps * L.wq;
    L.ws = xsw_region_bytes(x_bytes, max_m);
    L.red_off = L.xsum_off + kConsumerWarps * L.ws;
    L.info_off = L.red_off + red_bytes(max_m);
    L.bar_off = L.info_off + kInfoCap * 48;
    L.total = L.bar_off + kNumBars * 8 + 16;   // + abort flag
    return L;
}

__device__ __forceinline__ void red_release_gpu_add(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_gpu_add(int *p, int v) {
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_relaxed_gpu(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Bounded wait until *p >= want (GPU scope; acquire when the group was
// published with a release); false on timeout or abort.
__device__ __forceinline__ bool wait_count(const int *p, int want, bool acquire, uint64_t timeout_ns,
                                           const volatile int *abort_flag) {
    const uint64_t dl = global_timer() + timeout_ns;
    while ((acquire ? ld_acquire_gpu(p) : ld_relaxed_gpu(p)) < want) {
        if (*abort_flag || global_timer() > dl) return false;
    }
    return true;
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}
// The records are written into global memory by a host copy before the
// launch and rewritten between launches (the allocation-free entry point
// reuses one array for every call), while the TMA unit reads descriptors
// through the tensor-map proxy: the producer acquires each map, at system
// scope (the host wrote it), before its first use, so that no descriptor of
// an earlier call is used.  Measured cost: about 1% of a 225-matmul step.
__device__ __forceinline__ void acquire_tensormap(const CUtensorMap *m) {
    asm volatile("fence.proxy.tensormap::generic.acquire.sys [%0], 128;" ::"l"(m) : "memory");
}
__device__ __forceinline__ void acquire_record_maps(const ChainRec *r) {
    acquire_tensormap(&r->tw);
    acquire_tensormap(&r->ts);
    acquire_tensormap(&r->tb);
}

// The scalar part of a record (three 16-byte vectors).
struct RecInfo {
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    int M, N, K, T, flags, tile_base, bits, group;
};
__device__ __forceinline__ RecInfo unpack_info(uint4 a, uint4 b, uint4 c) {
    RecInfo i;
    i.x = reinterpret_cast<const __nv_bfloat16 *>((uint64_t)a.x | ((uint64_t)a.y << 32));
    i.y = reinterpret_cast<__nv_bfloat16 *>((uint64_t)a.z | ((uint64_t)a.w << 32));
    i.M = (int)b.x;
    i.N = (int)b.y;
    i.K = (int)b.z;
    i.T = (int)b.w;
    i.flags = (int)c.x;
    i.tile_base = (int)c.y;
    i.bits = (int)c.z;
    i.group = (int)c.w;
    return i;
}
// Record jm's scalars: the first kInfoCap come from the copy every CTA makes in
// shared memory at start (walking matmuls in which a CTA has no tile then costs
// no global-memory round trip), the rest from global memory.
__device__ __forceinline__ RecInfo load_info(const ChainRec *recs, const uint4 *info, int jm) {
    if (jm < kInfoCap) return unpack_info(info[3 * jm], info[3 * jm + 1], info[3 * jm + 2]);
    const uint4 *p = reinterpret_cast<const uint4 *>(&recs[jm].x);
    return unpack_info(__ldg(p), __ldg(p + 1), __ldg(p + 2));
}

// BITS: code width of every matmul of the chain (4 or 8); NV: every matmul
// holds NVFP4 weights (BITS = 4: same stage geometry, E4M3 block scales in
// place of the scale and bias boxes, no fold, the tensor scale applied by the
// reducer).
template <int BITS, bool ONE_ROW, bool NV = false>
__global__ void __launch_bounds__(kThreads, 1)
qmv_chain_kernel(const ChainRec *__restrict__ recs, int count, int *done, int x_bytes, int max_m,
                 unsigned long long timeout_ns, int *status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t s_base = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (s_base - raw_base);
    const ChainLayout L = chain_layout(x_bytes, max_m);
    const XStage xs = {s_base + (uint32_t)L.xq_off, s_base + (uint32_t)L.xsum_off, L.wq, L.ws};
    const uint32_t bar_full = s_base + L.bar_off;
    const uint32_t bar_empty = bar_full + kMaxStages * 8;
    const uint32_t bar_red = bar_empty + kMaxStages * 8;   // red_full[4], red_empty[4]
    constexpr int NS = kMaxStages;   // compile time: a runtime ring modulus measured 8% slower
    const uint32_t bar_dep = bar_red + 64;              // the previous matmul is complete (signaller -> consumers)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bar_off + kNumBars * 8);
    const int cta = (int)blockIdx.x, ncta = (int)gridDim.x;
    uint4 *info = reinterpret_cast<uint4 *>(smem + L.info_off);
    TileCtx tc;
    tc.red = reinterpret_cast<float *>(smem + L.red_off);
    tc.red_full = bar_red;
    tc.red_empty = bar_red + 32;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < 3 * (count < kInfoCap ? count : kInfoCap); i += blockDim.x)
        info[i] = __ldg(reinterpret_cast<const uint4 *>(&recs[i / 3].x) + i % 3);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        for (int p = 0; p < red_bufs<ONE_ROW>(); ++p) {
            mbar_init(tc.red_full + 8 * p, kConsumerWarps);
            mbar_init(tc.red_empty + 8 * p, 1);
        }
        mbar_init(bar_dep, 1);
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
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            bool ok = true;
            RecInfo cur = load_info(recs, info, 0);
            acquire_record_maps(recs);
            for (int jm = 0; jm < count && ok; ++jm) {
                const ChainRec *rec = recs + jm;
                // the next record's scalars and descriptors travel while this matmul streams
                RecInfo nxt = cur;
                if (jm + 1 < count) {
                    nxt = load_info(recs, info, jm + 1);
                    acquire_record_maps(rec + 1);
                    prefetch_tensormap(&rec[1].tw);
                    prefetch_tensormap(&rec[1].ts);
                    prefetch_tensormap(&rec[1].tb);
                }
                const int K = cur.K, T = cur.T;
                constexpr int SC = Geo<BITS>::kStageCodes, SG = Geo<BITS>::kStageGroups;
                const int KB = (K + SC - 1) / SC;
                // tiles are dealt round-robin, continuing from the previous
                // matmul of the same dependency group so that the group stays
                // balanced
                const int first = (cta - cur.tile_base % ncta + ncta) % ncta;
                for (int tile = first; tile < T && ok; tile += ncta) {
                    for (int kb = 0; kb < KB; ++kb) {
                        const int slot = issued % NS;
                        if (issued >= NS &&
                            !mbar_wait_for(bar_empty + 8 * slot, ((issued / NS) - 1) & 1, timeout_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if ((cur.flags & AQ_CHAIN_DEBUG_SKIP_COPY) && cta == 0 && tile == first && kb == 0) {
                            ++issued;   // test hook: this stage never arrives
                            continue;
                        }
                        const uint32_t dst = s_base + slot * kStageBytes;
                        const uint32_t fb = bar_full + 8 * slot;
                        // one copy of the stage's codes (chunks past the row's end read as zeros)
                        if (NV) {
                            // and one box of E4M3 scales: 128 bytes x 32 rows
                            mbar_expect_tx(fb, (uint32_t)kNvStage);
                            tma_load_3d(dst, &rec->tw, 0, tile * kRows, kb * kBoxes, fb, pol);
                            tma_load_2d(dst + kCodesBytes, &rec->ts, kb * (kNvCodes / 16), tile * kRows, fb, pol);
                        } else {
                            mbar_expect_tx(fb, (uint32_t)(kCodesBytes + 2 * kRows * SG * 2));
                            tma_load_3d(dst, &rec->tw, 0, tile * kRows, kb * kBoxes, fb, pol);
                            tma_load_2d(dst + kCodesBytes, &rec->ts, kb * SG, tile * kRows, fb, pol);
                            tma_load_2d(dst + kCodesBytes + kSBRegion, &rec->tb, kb * SG, tile * kRows, fb, pol);
                        }
                        ++issued;
                    }
                }
                cur = nxt;
            }
            if (!ok) {
                set_abort();
                const uint64_t drain = global_timer() + timeout_ns;
                for (int it = (issued > NS ? issued - NS : 0); it < issued; ++it)
                    while (!mbar_try_wait(bar_full + 8 * (it % NS), (it / NS) & 1) && global_timer() < drain) {
                    }
            }
        }
        __syncwarp();
    } else if (warp == kConsumerWarps + 1) {
        // ------------------------------------------------------------ reducer / signaller
        // Adds the sixteen warps' partials of each of this CTA's tiles in order
        // and stores y.  A dependency group is a dependent matmul and the
        // independent ones after it; each has one completion counter.  After
        // the CTA's last tile of a group the warp publishes its tile count of
        // the group (one GPU-scope release per CTA and group, off the
        // consumers' path); before a dependent matmul it waits until every CTA
        // has stored all tiles of the previous group, then releases the
        // consumers.
        int tcount = 0, pending = 0;
        bool ok = true;
        RecInfo prev = load_info(recs, info, 0), cur = prev;
        for (int jm = 0; jm < count; ++jm) {
            RecInfo nxt = cur;
            if (jm + 1 < count) nxt = load_info(recs, info, jm + 1);
            if (jm > 0 && !(cur.flags & AQ_CHAIN_INDEPENDENT)) {
                if (lane == 0) {
                    // the previous group's tiles: its last matmul's tile_base counts the ones before it
                    const int want = prev.tile_base + prev.T;
                    if (ok && !wait_count(done + prev.group, want, (prev.flags & kRecRelease) != 0, timeout_ns,
                                          abort_flag)) {
                        set_abort();
                        ok = false;
                    }
                    mbar_arrive(bar_dep);
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            }
            const int first = (cta - cur.tile_base % ncta + ncta) % ncta;
            float yscale = 1.f;
            if (NV && first < cur.T) {
                const float *gs = recs[jm].gscale;
                yscale = __ldg(gs);
            }
            for (int tile = first; tile < cur.T && ok; tile += ncta, ++pending, ++tcount)
                ok = reduce_tile<ONE_ROW>(tc, tcount, tile, cur.M, cur.N, cur.y, lane, timeout_ns, abort_flag, nullptr,
                                          0, 1, yscale);
            const bool group_ends = jm + 1 == count || !(nxt.flags & AQ_CHAIN_INDEPENDENT);
            if (ok && group_ends && pending > 0 && lane == 0) {
                // every lane's y stores precede this (reduce_tile ends with __syncwarp);
                // where a later matmul touches what this group wrote, the release
                // makes them visible at GPU scope before the count
                if (cur.flags & kRecRelease)
                    red_release_gpu_add(done + cur.group, pending);
                else
                    red_relaxed_gpu_add(done + cur.group, pending);
            }
            if (group_ends) pending = 0;
            if (!ok && lane == 0) set_abort();
            prev = cur;
            cur = nxt;
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- consumers
        // Each warp stages its own slice of each new x (no barrier with the
        // other warps) and runs the tiles over its column blocks; after an
        // abort the remaining matmuls are walked through without work.
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float inv[2] = {1.f, 1.f};
        int tcount = 0, item = 0, ndep = 0;
        bool ok = true;
        const __nv_bfloat16 *prev_x = nullptr;
        int prev_M = 0, prev_K = 0, prev_bits = 0;
        RecInfo cur = load_info(recs, info, 0);
        for (int jm = 0; jm < count; ++jm) {
            RecInfo nxt = cur;
            if (jm + 1 < count) nxt = load_info(recs, info, jm + 1);
            const int M = cur.M, K = cur.K, T = cur.T;
            // A matmul flagged independent does not read the previous one's
            // output: it neither waits for it nor, when its x is the same
            // buffer (staged for the same code width), reloads x.
            const bool dep = jm > 0 && !(cur.flags & AQ_CHAIN_INDEPENDENT);
            const bool new_x = jm == 0 || cur.x != prev_x || M != prev_M || K != prev_K || cur.bits != prev_bits;
            if (dep) {
                // the signaller saw every tile of matmul jm-1 stored
                if (ok && !mbar_wait_for(bar_dep, (uint32_t)(ndep & 1), timeout_ns, abort_flag)) ok = false;
                ++ndep;
            }
            prev_x = cur.x;
            prev_M = M;
            prev_K = K;
            prev_bits = cur.bits;

            if (NV) {
                const int nblk = K / 128;
                const int KB = (K + kNvCodes - 1) / kNvCodes;
                if (new_x && ok) stage_x_nv_warp<ONE_ROW>(xs, cur.x, M, K, warp, lane, inv);
                NvThread ct;
                nv_consumer_init(ct, warp, lane);
                // the lane's x: row lane/4 (B column lane/4), fragment t = lane % 4
                const int M1 = ONE_ROW ? 1 : M, xrow = ONE_ROW ? 0 : ((lane >> 2) < M1 ? (lane >> 2) : M1 - 1);
                const uint32_t xq = xs.xq + (uint32_t)(warp * xs.wq + xrow * xw_row_bytes(M1, KB, 4) + (lane & 3) * 8);
                const int first = (cta - cur.tile_base % ncta + ncta) % ncta;
                for (int tile = first; tile < T && ok; tile += ncta) {
                    for (int kb = 0; kb < KB; ++kb, ++item) {
                        const int slot = item % NS;
                        const uint32_t phase = (uint32_t)(item / NS) & 1u;
                        if (!mbar_wait_for(bar_full + 8 * slot, phase, timeout_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (kb * kConsumerWarps + warp < nblk)
                            consume_stage_nvfp4(s_base + (uint32_t)(slot * kStageBytes), ct, xq + (uint32_t)(kb * 256), acc);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
                    }
                    if (!ok) break;
                    ok = deposit_tile<ONE_ROW>(tc, acc, tcount, M, warp, lane, lane >> 2, inv, timeout_ns,
                                               abort_flag);
                    ++tcount;
                }
            } else {
                using Gm = Geo<BITS>;
                const int nblk = K / Gm::kWarpCodes;
                const int KB = (K + Gm::kStageCodes - 1) / Gm::kStageCodes;
                // ---- this warp's slice of x: L2 loads, fp16 fragments, group sums and scale
                if (new_x && ok) stage_x_warp<BITS, ONE_ROW>(xs, cur.x, M, K, K, warp, lane, inv);

                ConsumerThread ct;
                consumer_init<BITS, ONE_ROW>(ct, warp, lane, xs, M, K);

                const int first = (cta - cur.tile_base % ncta + ncta) % ncta;
                for (int tile = first; tile < T && ok; tile += ncta) {
                    for (int kb = 0; kb < KB; ++kb, ++item) {
                        const int slot = item % NS;
                        const uint32_t phase = (uint32_t)(item / NS) & 1u;
                        if (!mbar_wait_for(bar_full + 8 * slot, phase, timeout_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (kb * kConsumerWarps + warp < nblk)
                            consume_stage<BITS, ONE_ROW>(s_base + (uint32_t)(slot * kStageBytes), kb, ct, acc);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
                    }
                    if (!ok) break;
                    ok = deposit_tile<ONE_ROW>(tc, acc, tcount, M, warp, lane, lane >> 2, inv, timeout_ns,
                                               abort_flag);
                    ++tcount;
                }
            }
            if (!ok) set_abort();   // the remaining matmuls are walked through without work
            cur = nxt;
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

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int kMaxDevices = 64;
std::atomic<int> g_attr_done[6][kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];

size_t records_bytes(int count) { return (size_t)count * sizeof(ChainRec); }
size_t counters_bytes(int count) { return ((size_t)count * sizeof(int) + 127) & ~(size_t)127; }

}  // namespace

size_t chain_workspace_bytes(int count) {
    if (count <= 0) return 0;
    return records_bytes(count) + counters_bytes(count);
}

namespace {

// The chain's weight format: affine codes of 4 or 8 bits in groups of 64, or
// NVFP4 (group size 16: E2M1 codes, E4M3 block scales, a tensor scale).
bool chain_format_ok(int group_size, int bits) {
    return (group_size == 64 && (bits == 4 || bits == 8)) || (group_size == 16 && bits == 4);
}

// Validates the descriptors (host only, no CUDA call).
aq_status chain_validate(const aq_matmul_desc *descs, int count, int group_size, int bits) {
    if (!chain_format_ok(group_size, bits)) return AQ_ERR_UNSUPPORTED;
    const bool nv = group_size == 16;
    for (int i = 0; i < count; ++i) {
        const aq_matmul_desc &d = descs[i];
        if (d.M < 1 || d.N < 1 || d.K < 1 || d.K % group_size) return AQ_ERR_INVALID_ARG;
        if (d.flags & ~(int64_t)(AQ_CHAIN_INDEPENDENT | AQ_CHAIN_RELEASE | AQ_CHAIN_DEBUG_SKIP_COPY))
            return AQ_ERR_INVALID_ARG;
        if (!d.x || !d.w_packed || !d.scales || !d.biases || !d.y) return AQ_ERR_INVALID_ARG;
        // affine: K in whole 512-code chunks (16-byte rows of scales); NVFP4: 256 (16-byte scale rows)
        if (d.M > 8 || d.K % (nv ? 256 : 512) || d.K > (int64_t)1 << 20 || d.N > (int64_t)1 << 30)
            return AQ_ERR_UNSUPPORTED;
        if (x_stage_bytes((int)d.M, (int)d.K, bits) > kMaxXBytes) return AQ_ERR_UNSUPPORTED;
        if (!aligned(d.x, 16) || !aligned(d.w_packed, 16) || !aligned(d.scales, 16) ||
            !aligned(d.biases, nv ? 4 : 16) || !aligned(d.y, 2))
            return AQ_ERR_ALIGNMENT;
    }
    return AQ_OK;
}

// Byte ranges a matmul reads (x, codes, scales, biases or the NVFP4 tensor
// scale) and writes (y).
struct Footprint {
    uintptr_t r[4][2];
    uintptr_t w[2];
};
Footprint footprint(const aq_matmul_desc &d, int bits, bool nv) {
    auto range = [](const void *p, uint64_t n, uintptr_t (&o)[2]) {
        o[0] = reinterpret_cast<uintptr_t>(p);
        o[1] = o[0] + n;
    };
    const uint64_t M = (uint64_t)d.M, N = (uint64_t)d.N, K = (uint64_t)d.K;
    Footprint f;
    range(d.x, M * K * 2, f.r[0]);
    range(d.w_packed, N * K * (uint64_t)bits / 8, f.r[1]);
    range(d.scales, nv ? N * K / 16 : N * (K / 64) * 2, f.r[2]);
    range(d.biases, nv ? 4 : N * (K / 64) * 2, f.r[3]);
    range(d.y, M * N * 2, f.w);
    return f;
}
// Marks, on the last matmul of each dependency group, whether its completion
// is published with a release (kRecRelease): where a hazard pair (i, k), i <=
// the group's last matmul < k, crosses it, or where the caller asks for it
// (AQ_CHAIN_RELEASE on any of the group's matmuls).  Every group a hazard
// crosses is marked, so the release / acquire pairs chain from i to k.  The
// last group's completion is never awaited inside the chain (the kernel's
// end orders it for later work).
//
// The pairs come from one sweep over every byte range of the chain sorted by
// start (O(n log n) plus the overlapping pairs); past kPairBudget overlapping
// pairs (chains whose matmuls share much memory) every group is released.
constexpr long kPairBudget = 1L << 22;
struct Span {
    uintptr_t lo, hi;
    int mm;
    bool write;
};
// Working room of mark_releases for `count` matmuls: spans and active hold 5 *
// count entries, latest count, cover count + 1 (the caller provides it, so that
// the allocation-free entry point can pass static arrays).
struct ReleaseScratch {
    Span *spans;
    int *active, *latest, *cover;
};
void mark_releases(const aq_matmul_desc *descs, int count, int bits, bool nv, ChainRec *recs,
                   const ReleaseScratch &w) {
    int ns = 0;
    for (int i = 0; i < count; ++i) {
        const Footprint f = footprint(descs[i], bits, nv);
        for (int a = 0; a < 4; ++a)
            if (f.r[a][1] > f.r[a][0]) w.spans[ns++] = {f.r[a][0], f.r[a][1], i, false};
        if (f.w[1] > f.w[0]) w.spans[ns++] = {f.w[0], f.w[1], i, true};
    }
    std::sort(w.spans, w.spans + ns, [](const Span &a, const Span &b) { return a.lo < b.lo; });
    for (int i = 0; i < count; ++i) w.latest[i] = -1;   // latest k > i with a hazard against matmul i
    int na = 0;                                         // spans still open at the current start
    long pairs = 0;
    bool all = false;
    for (int s = 0; s < ns && !all; ++s) {
        const Span &cur = w.spans[s];
        int kept = 0;
        for (int a = 0; a < na; ++a)
            if (w.spans[w.active[a]].hi > cur.lo) w.active[kept++] = w.active[a];   // overlaps cur
        na = kept;
        for (int a = 0; a < na; ++a) {
            const Span &o = w.spans[w.active[a]];
            if ((o.write || cur.write) && o.mm != cur.mm) {
                const int i = std::min(o.mm, cur.mm), k = std::max(o.mm, cur.mm);
                w.latest[i] = std::max(w.latest[i], k);
            }
            if (++pairs > kPairBudget) all = true;
        }
        w.active[na++] = s;
    }
    for (int j = 0; j <= count; ++j) w.cover[j] = 0;   // difference array over matmul positions
    if (all) {
        w.cover[0] = 1;
    } else {
        for (int i = 0; i < count; ++i)
            if (w.latest[i] > i) {
                ++w.cover[i];
                --w.cover[w.latest[i]];
            }
    }
    int run = 0;
    bool forced = false;
    for (int j = 0; j < count; ++j) {
        run += w.cover[j];
        forced = forced || (descs[j].flags & AQ_CHAIN_RELEASE) != 0;
        const bool group_end = j + 1 == count || !(descs[j + 1].flags & AQ_CHAIN_INDEPENDENT);
        if (!group_end) continue;
        if (j + 1 < count && (run > 0 || forced)) recs[j].flags |= kRecRelease;
        forced = false;
    }
}

// Encodes validated descriptors into host records and fills the plan's sizes.
aq_status chain_encode(const aq_matmul_desc *descs, int count, int group_size, int bits, ChainRec *recs,
                       aq_chain_plan *plan, const ReleaseScratch &scratch) {
    if (!encode_fn()) return AQ_ERR_UNSUPPORTED;
    const bool nv = group_size == 16;
    int x_bytes = 16;
    bool one_row = true;
    for (int i = 0; i < count; ++i) {
        const aq_matmul_desc &d = descs[i];
        ChainRec &r = recs[i];
        std::memset(&r, 0, sizeof r);
        const uint64_t K = (uint64_t)d.K, N = (uint64_t)d.N, G = K / 64;
        // codes: one stage (8 chunks x 32 rows x 128 bytes, 128-byte swizzle) per box; scales
        // and biases: one stage's groups x 32 rows (64-byte rows and swizzle for 4-bit codes,
        // 32 for 8-bit)
        const uint32_t sg = (uint32_t)stage_groups(bits);
        const CUtensorMapSwizzle sbs = bits == 8 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
        if (nv) {
            // NVFP4: E4M3 scales [N][K/16] bytes, one 128-byte x 32-row box per stage (128-byte swizzle)
            if (!encode_codes_3d(&r.tw, d.w_packed, K / 2, N) ||
                !encode_2d(&r.ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, d.scales, K / 16, N, K / 16, kNvCodes / 16, kRows,
                           CU_TENSOR_MAP_SWIZZLE_128B))
                return AQ_ERR_INVALID_ARG;
            r.tb = r.ts;   // a valid map in the unused slot (the producer acquires all three)
            r.gscale = static_cast<const float *>(d.biases);
        } else if (!encode_codes_3d(&r.tw, d.w_packed, K * bits / 8, N) ||
                   !encode_2d(&r.ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, d.scales, G, N, G * 2, sg, kRows, sbs) ||
                   !encode_2d(&r.tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, d.biases, G, N, G * 2, sg, kRows, sbs)) {
            return AQ_ERR_INVALID_ARG;
        }
        r.x = static_cast<const __nv_bfloat16 *>(d.x);
        r.y = static_cast<__nv_bfloat16 *>(d.y);
        r.M = (int)d.M;
        r.N = (int)d.N;
        r.K = (int)d.K;
        r.tiles = (int)((d.N + kRows - 1) / kRows);
        r.flags = (int)d.flags;
        r.bits = bits;
        const bool indep = i > 0 && (d.flags & AQ_CHAIN_INDEPENDENT);
        r.tile_base = indep ? recs[i - 1].tile_base + recs[i - 1].tiles : 0;
        r.group = indep ? recs[i - 1].group : i;
        x_bytes = std::max(x_bytes, x_stage_bytes((int)d.M, (int)d.K, bits));
        one_row = one_row && d.M == 1;
    }
    plan->count = count;
    plan->x_bytes = (x_bytes + 15) & ~15;
    plan->one_row = one_row ? 1 : 0;
    plan->reserved[0] = bits;   // code width of the chain (selects the kernel)
    plan->reserved[2] = nv ? 1 : 0;   // NVFP4 weights
    for (int i = 0; i < count; ++i)
        if (descs[i].flags & AQ_CHAIN_DEBUG_SKIP_COPY) plan->reserved[1] = 1;   // the test hook: short waits
    mark_releases(descs, count, bits, nv, recs, scratch);
    for (int i = 0; i < count; ++i)
        if (recs[i].flags & kRecRelease) ++plan->reserved[3];   // groups published with a release
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
    if (!chain_format_ok(group_size, bits)) return AQ_ERR_UNSUPPORTED;
    if (workspace_bytes < chain_workspace_bytes(count)) return AQ_ERR_INVALID_ARG;
    if (!aligned(workspace, 128)) return AQ_ERR_ALIGNMENT;
    aq_status st = chain_validate(descs, count, group_size, bits);  // before any CUDA call
    if (st != AQ_OK) return st;
    std::vector<ChainRec> recs((size_t)count);
    std::vector<Span> spans((size_t)count * 5);
    std::vector<int> active((size_t)count * 5), latest((size_t)count), cover((size_t)count + 1);
    const ReleaseScratch scratch = {spans.data(), active.data(), latest.data(), cover.data()};
    st = chain_encode(descs, count, group_size, bits, recs.data(), plan, scratch);
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
    if (plan->reserved[1]) timeout_ns = 20000000ull;   // the test hook: 20 ms waits
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
    const int count = plan->count;
    const int max_m = plan->one_row ? 1 : kMaxM;
    const ChainLayout L = chain_layout(plan->x_bytes, max_m);
    const int smem = L.total + 1024;
    const bool one = plan->one_row != 0;
    const bool eight = plan->reserved[0] == 8, nv = plan->reserved[2] != 0;
    auto kern = nv      ? (one ? qmv_chain_kernel<4, true, true> : qmv_chain_kernel<4, false, true>)
                : eight ? (one ? qmv_chain_kernel<8, true> : qmv_chain_kernel<8, false>)
                        : (one ? qmv_chain_kernel<4, true> : qmv_chain_kernel<4, false>);
    const int ki = nv ? 4 + (int)one : 2 * (int)eight + (int)one;
    if (!g_attr_done[ki][dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemLimit);
        if (e != cudaSuccess) return e;
        g_attr_done[ki][dev].store(1, std::memory_order_release);
    }
    int *done = reinterpret_cast<int *>(static_cast<uint8_t *>(plan->workspace) + records_bytes(count));
    e = cudaMemsetAsync(done, 0, counters_bytes(count), stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sms);   // one CTA per SM, all resident (they wait on one another)
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const ChainRec *>(plan->workspace), count, done, plan->x_bytes,
                              max_m, (unsigned long long)timeout_ns, status);
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
Span g_static_spans[5 * kStaticChainMax];       // and the release marking's working room
int g_static_active[5 * kStaticChainMax], g_static_latest[kStaticChainMax], g_static_cover[kStaticChainMax + 1];
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
    // The host staging array is shared too, and the record copy, the counter
    // clear and the launch of one call must reach the stream together: two
    // host threads enqueueing on one stream would otherwise interleave them
    // (one call's kernel running the other's records).  So the lock covers
    // all three.
    std::lock_guard<std::mutex> lock(g_static_host_mutex);
    const ReleaseScratch marks = {g_static_spans, g_static_active, g_static_latest, g_static_cover};
    st = chain_encode(descs, count, group_size, bits, g_static_host_recs, &plan, marks);
    if (st != AQ_OK) return st;
    // from pageable memory: returns once the records are staged (which may
    // mean waiting for the stream's earlier work), so the host array may be
    // reused by the next call
    *err = cudaMemcpyAsync(scratch, g_static_host_recs, records_bytes(count), cudaMemcpyHostToDevice, stream);
    if (*err != cudaSuccess) return AQ_ERR_CUDA;
    plan.workspace = scratch;
    *err = chain_run(&plan, timeout_ns, status, stream);  // clears the counters, then launches
    return *err == cudaSuccess ? AQ_OK : AQ_ERR_CUDA;
}

}  // namespace aq
