// Weight-streaming kernel for y = x . dequant(W)^T with 1..8 rows of x,
// fed by the Tensor Memory Accelerator.
//
// Decode time is the time to stream the packed weights ("epic: CUDA (MLX
// backend) prefill and decode acceleration program", Diagnosis; "gemma-4
// decode carries ~44 ms/token ...", re-scope paragraph).  This kernel keeps
// the weight stream going independently of the arithmetic:
//
//  * one producer warp per CTA copies 32-row x 2048-code tiles of the packed
//    codes, plus the matching scales and biases, into a ring of shared-memory
//    stages with cp.async.bulk.tensor (TMA), completion tracked by mbarriers;
//  * sixteen consumer warps each take one 128-code column block of a stage
//    (32 rows x 2 groups) and run the dequantization-free dot product of the
//    folded form on mma.sync m16n8k16 (fp16 in, fp32 out), with the codes as
//    exact fp16 values 1024 + q and x staged as fp16 fragments, each warp
//    loading and converting only the slice of x its column blocks use, with
//    no barrier against the other warps (qmv_consumer.cuh has the arithmetic
//    and its exactness argument);
//  * CTAs are persistent, one per SM: each walks its 32-row tiles across the
//    whole K, the sixteen warps' partial sums are combined in shared memory
//    in a fixed order, and every output is written exactly once
//    (deterministic).  One CTA of sixteen consumer warps (rather than two of
//    eight) lets a single tile use the whole SM, which matters for matrices
//    with fewer tiles than twice the SM count.
//
// A warp covers 32 rows so that each x fragment it loads feeds two MMAs: the
// consumer is bound by shared-memory bandwidth, and the x fragments are the
// largest part of it.  The code tiles use the TMA 128-byte swizzle and the
// scale/bias tiles the 64-byte swizzle, so the consumers' shared-memory reads
// are free of bank conflicts.
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

constexpr int kReducers = 2;   // reducer warps, each summing half the rows of every tile
constexpr int kThreads = (kConsumerWarps + 1 + kReducers) * 32;   // consumers, TMA producer, reducers
constexpr int kMaxStages = 4;   // ring depth (36 KB stages); 5 measured no faster
constexpr int kNumBars = 2 * kMaxStages + 8;   // full[S], empty[S], red_full[4], red_empty[4]
constexpr int kSmemLimit = 232448;               // dynamic shared memory a CTA may use

struct Layout {
    int stages;      // ring depth (kMaxStages)
    int xq_off;      // per-warp fragment regions of the staged x (one K pass), wq bytes each
    int wq;
    int xsum_off;    // per-warp (Xs, X') regions, ws bytes each
    int ws;
    int red_off;     // float [bufs][16][32][M]
    int yacc_off;    // float [cap][32][M]: tile sums across K passes (when there are several)
    int bar_off;     // uint64 [kNumBars] + abort flag
    int total;       // bytes (excluding the 1024 alignment slack)
};
// Kp: codes of K per pass; cap: tiles per batch kept in yacc (0 with one pass)
// ns: ring depth (4, or 3 to make room for x of up to 64 KB in one pass)
__host__ __device__ inline Layout make_layout(int M, int Kp, int cap, int bits, int ns = kMaxStages) {
    Layout L;
    const int xb = x_stage_bytes(M, Kp, bits);
    L.stages = ns;
    L.xq_off = L.stages * kStageBytes;
    L.wq = xw_region_bytes(xb, M);
    L.xsum_off = L.xq_off + kConsumerWarps * L.wq;
    L.ws = xsw_region_bytes(xb, M);
    L.red_off = L.xsum_off + kConsumerWarps * L.ws;
    L.yacc_off = L.red_off + red_bytes(M);
    L.bar_off = L.yacc_off + cap * kRows * M * 4;
    L.total = L.bar_off + kNumBars * 8 + 16;
    return L;
}
constexpr int kMaxSmem = kSmemLimit;

// BITS: code width (4 or 8).  ONE_ROW: M == 1 (every MMA column holds x row 0).
// One CTA per SM.  MULTI: x (M x K) is larger than one staging (M*K*2 >
// 32 KB), so K is walked in passes of Kp codes (kbp stages): the CTA's tiles
// go in batches of `cap`, and for each batch every pass stages its slice of x
// and runs the batch's tiles over the pass's stages; the reducer keeps the
// tile sums across passes.  Each weight byte is still read once.  Without
// MULTI, x is staged once (kbp and cap are unused).
// skip_copy: test hook; the producer leaves out the first stage's copies, so the
// consumers' bounded wait on it expires.
// NS: ring depth; 3 leaves room for x of up to 64 KB (one pass for, e.g., 8 rows of K = 4096).
// NB: blocks of 8 MMA columns, 2 for 9..16 rows of x (every code pair feeds both).
// split_rows: CTAs 2p and 2p + 1 take rows [0, ceil(M/2)) and [ceil(M/2), M) of x
// and y and walk the same tiles at the same pace, so that the second copy of a
// tile mostly finds it in L2 (9..16 rows as two halves of at most 8 in one launch).
template <int BITS, bool ONE_ROW, bool MULTI, int NS = kMaxStages, int NB = 1>
__global__ void __launch_bounds__(kThreads, 1)
qmv_tma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
               const __grid_constant__ CUtensorMap tm_b, const __nv_bfloat16 *__restrict__ x,
               __nv_bfloat16 *__restrict__ y, int M, int N, int K, int kbp, int cap, unsigned long long timeout_ns,
               int *status, int skip_copy, int split_rows) {
    using Gm = Geo<BITS>;
    // the CTA's place among those walking the tiles (a pair counts once with split_rows;
    // the two-block instances never split, and keep x, y and M as launched)
    const bool split = NB == 1 && split_rows;
    const int cta = split ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int ncta = split ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    if (split) {
        const int half = (int)(blockIdx.x & 1u), m0 = half ? (M + 1) / 2 : 0;
        x += (size_t)m0 * K;
        y += (size_t)m0 * N;
        M = half ? M / 2 : (M + 1) / 2;
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int KB = (K + Gm::kStageCodes - 1) / Gm::kStageCodes;    // stages per tile
    if (!MULTI) kbp = KB;
    const int P = MULTI ? (KB + kbp - 1) / kbp : 1;                // K passes
    const int Kp = MULTI ? kbp * Gm::kStageCodes : K;
    const Layout L = make_layout(M, Kp, MULTI ? cap : 0, BITS, NS);
    const uint32_t s_base = smem_addr(smem);
    // NS at compile time: a runtime ring modulus measured 8% slower
    constexpr int kXRoom = NS == kMaxStages ? kMaxXBytes : 2 * kMaxXBytes;
    const XStage xs = {s_base + (uint32_t)L.xq_off, s_base + (uint32_t)L.xsum_off, L.wq, L.ws};
    float *yacc = reinterpret_cast<float *>(smem + L.yacc_off);
    const uint32_t bar_full = s_base + L.bar_off;          // NS barriers (room for kMaxStages)
    const uint32_t bar_empty = bar_full + kMaxStages * 8;  // NS barriers
    const uint32_t bar_red = bar_empty + kMaxStages * 8;   // red_full[4], red_empty[4]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bar_off + kNumBars * 8);
    TileCtx tc;
    tc.red = reinterpret_cast<float *>(smem + L.red_off);
    tc.red_full = bar_red;
    tc.red_empty = bar_red + 32;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = (N + kRows - 1) / kRows;
    const int my_tiles = cta < T ? (T - 1 - cta) / ncta + 1 : 0;
    const int L_items = my_tiles * KB;
    if (!MULTI) cap = my_tiles > 0 ? my_tiles : 1;   // one batch

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        for (int p = 0; p < red_bufs<ONE_ROW, NB>(); ++p) {
            mbar_init(tc.red_full + 8 * p, kConsumerWarps);
            mbar_init(tc.red_empty + 8 * p, kReducers);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    griddep_launch();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // stage order: tile batches, K passes, the batch's tiles, the pass's stages
            int tb = 0, p = 0, t = 0, kb = 0;
            auto advance = [&]() {
                const int kb1 = (p + 1) * kbp < KB ? (p + 1) * kbp : KB;
                if (++kb < kb1) return;
                kb = p * kbp;
                const int tb_end = tb + cap < my_tiles ? tb + cap : my_tiles;
                if (++t < tb_end) return;
                t = tb;
                if (++p < P) {
                    kb = p * kbp;
                    return;
                }
                p = 0;
                tb += cap;
                t = tb;
                kb = 0;
            };
            auto issue = [&](int it) {
                const int slot = it % NS;
                const int tile = cta + t * ncta;
                const uint32_t dst = s_base + slot * kStageBytes;
                const uint32_t fb = bar_full + 8 * slot;
                if (skip_copy && it == 0) {   // test hook: this stage never arrives
                    advance();
                    return;
                }
                // one box of 8 chunks x 32 rows x 128 bytes (chunks past the row's end read as
                // zeros and still count toward the transaction)
                mbar_expect_tx(fb, (uint32_t)(kCodesBytes + 2 * kRows * Gm::kSBRowBytes));
                tma_load_3d(dst, &tm_w, 0, tile * kRows, kb * kBoxes, fb, pol);
                tma_load_2d(dst + kCodesBytes, &tm_s, kb * Gm::kStageGroups, tile * kRows, fb, pol);
                tma_load_2d(dst + kCodesBytes + kSBRegion, &tm_b, kb * Gm::kStageGroups, tile * kRows, fb, pol);
                advance();
            };
            int issued = 0;
            bool ok = true;
            // the weights do not depend on the preceding kernel: prefetch them first
            for (; issued < L_items && issued < NS; ++issued) issue(issued);
            const uint64_t deadline = global_timer() + timeout_ns;
            for (; issued < L_items; ++issued) {
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
                // let the copies already issued land before the CTA can exit
                const uint64_t drain = global_timer() + timeout_ns;
                for (int it = (issued > NS ? issued - NS : 0); it < issued; ++it)
                    while (!mbar_try_wait(bar_full + 8 * (it % NS), (it / NS) & 1) && global_timer() < drain) {
                    }
            }
        }
        __syncwarp();
    } else if (warp > kConsumerWarps) {
        // ------------------------------------------------------------ reducers
        // Add the sixteen warps' partials of each tile and store y (the
        // consumers deposit a tile only after their griddepcontrol.wait, so y
        // is written after the preceding kernel).  Reducer r takes rows
        // [r, r + 1) * 32 / kReducers of every tile, and with K passes it
        // keeps those rows' sums across the passes.
        const int r = warp - kConsumerWarps - 1;
        int tcount = 0;
        bool ok = true;
        if (!MULTI) {
            for (int t = 0; ok && t < my_tiles; ++t, ++tcount)
                ok = reduce_tile<ONE_ROW, NB>(tc, tcount, cta + t * ncta, M, N, y, lane,
                                              timeout_ns, abort_flag, nullptr, 0, 1, 1.f, r, kReducers);
        } else {
            for (int tb = 0; ok && tb < my_tiles; tb += cap) {
                const int tb_end = tb + cap < my_tiles ? tb + cap : my_tiles;
                for (int p = 0; ok && p < P; ++p)
                    for (int t = tb; ok && t < tb_end; ++t, ++tcount)
                        ok = reduce_tile<ONE_ROW, NB>(tc, tcount, cta + t * ncta, M, N, y,
                                                      lane, timeout_ns, abort_flag, yacc + (t - tb) * kRows * M, p, P,
                                                      1.f, r, kReducers);
            }
        }
        if (!ok && lane == 0 && !*abort_flag) {
            atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ---------------------------------------------------------------- consumers
        // Each warp stages its own slice of x (no barrier with the other warps)
        // and runs every tile over its column blocks; after an abort the waits
        // return at once and the work is skipped.
        griddep_wait();  // x comes from the preceding kernel; the deadline starts after it
        const uint64_t deadline = global_timer() + timeout_ns;
        float acc[NB][2][4] = {};
        float inv[2 * NB];
        bool ok = !*abort_flag;
        int item = 0, tcount = 0;
        // one tile over stages [kb0, kb1) of the staged slice of x, then its partials to the reducer
        auto run_tile = [&](const ConsumerThread &ct, int kb0, int kb1, int nblk) {
            for (int kb = kb0; ok && kb < kb1; ++kb, ++item) {
                const int slot = item % NS;
                if (!mbar_wait_fast(bar_full + 8 * slot, (uint32_t)(item / NS) & 1u, deadline, abort_flag)) {
                    ok = false;
                    break;
                }
                if ((kb - kb0) * kConsumerWarps + warp < nblk) {
                    if constexpr (NB == 2)
                        consume_stage2<BITS>(s_base + (uint32_t)(slot * kStageBytes), kb - kb0, ct, acc);
                    else
                        consume_stage<BITS, ONE_ROW>(s_base + (uint32_t)(slot * kStageBytes), kb - kb0, ct, acc[0]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
            }
            if (ok) {
                if constexpr (NB == 2)
                    ok = deposit_tile2(tc, acc, tcount, M, warp, lane, inv, timeout_ns, abort_flag);
                else
                    ok = deposit_tile<ONE_ROW>(tc, acc[0], tcount, M, warp, lane, lane >> 2, inv, timeout_ns,
                                               abort_flag);
            }
            ++tcount;
        };
        if (!MULTI) {
            stage_x_warp<BITS, ONE_ROW, kXRoom, NB>(xs, x, M, K, K, warp, lane, inv);
            ConsumerThread ct;
            consumer_init<BITS, ONE_ROW, NB>(ct, warp, lane, xs, M, K);
            for (int t = 0; t < my_tiles; ++t) run_tile(ct, 0, KB, K / Gm::kWarpCodes);
        } else {
            for (int tb = 0; tb < my_tiles; tb += cap) {
                const int tb_end = tb + cap < my_tiles ? tb + cap : my_tiles;
                for (int p = 0; p < P; ++p) {
                    const int k0 = p * Kp, Kpass = K - k0 < Kp ? K - k0 : Kp;
                    const int kb0 = p * kbp, kb1 = kb0 + kbp < KB ? kb0 + kbp : KB;
                    // the pass's slice of x, from L2
                    stage_x_warp<BITS, ONE_ROW, kXRoom, NB>(xs, x + k0, M, Kpass, K, warp, lane, inv);
                    ConsumerThread ct;
                    consumer_init<BITS, ONE_ROW, NB>(ct, warp, lane, xs, M, Kpass);
                    for (int t = tb; t < tb_end; ++t) run_tile(ct, kb0, kb1, Kpass / Gm::kWarpCodes);
                }
            }
        }
        if (!ok && lane == 0 && !*abort_flag) {
            atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
            *abort_flag = 1;
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
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_attr_done[32][kMaxDevices];

}  // namespace

// The packed codes as a 3-D tensor {32 words, N rows, row bytes / 128 chunks} (the
// chunks 128 bytes apart, rows row_bytes apart), read in boxes of {32, 32, 8}:
// one copy brings a whole stage, laid out as 8 chunk planes of 32 rows x 128
// bytes with the 128-byte swizzle.
bool encode_codes_3d(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {32, rows, row_bytes / 128};
    cuuint64_t strides[2] = {row_bytes, 128};
    cuuint32_t box[3] = {32, (cuuint32_t)kRows, (cuuint32_t)kBoxes};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return encode_fn(); }

bool qmv_tma_supported(const MatmulArgs &a) {
    return (a.bits == 4 || a.bits == 8) && a.M >= 1 && a.M <= kMaxRows && a.K % 512 == 0 && encode_fn() != nullptr &&
           (reinterpret_cast<uintptr_t>(a.scales) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.biases) & 15) == 0;
}

namespace {
// stages of K per pass: as many whole stages as keep one pass of x within kMaxXBytes
// x within kMaxXBytes is staged beside a 4-stage ring; larger x gets twice the
// room beside a 3-stage ring, in one pass where it fits (8 rows of K = 4096:
// lm_head 92 -> 60 us against two passes), else in passes of as many whole
// stages as fit.
int ring_stages(int M, int K, int bits) { return x_stage_bytes(M, K, bits) <= kMaxXBytes ? kMaxStages : 3; }
int x_room(int ns) { return ns == kMaxStages ? kMaxXBytes : 2 * kMaxXBytes; }
int stages_per_pass(int M, int K, int bits) {
    return std::max(1, x_room(ring_stages(M, K, bits)) / 2 / M / stage_codes(bits));
}
}  // namespace

int qmv_tma_passes(const MatmulArgs &a) {
    const int SC = stage_codes(a.bits), kbp = stages_per_pass((int)a.M, (int)a.K, a.bits);
    const int KB = (int)((a.K + SC - 1) / SC);
    return (KB + kbp - 1) / kbp;
}

namespace {
cudaError_t device_sms(int *dev, int *sms) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
    *sms = g_sms[*dev].load(std::memory_order_relaxed);
    if (*sms == 0) {
        e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess) return e;
        g_sms[*dev].store(*sms, std::memory_order_relaxed);
    }
    return cudaSuccess;
}
}  // namespace

// Measured on GB300 against the general kernel (graph-replayed calls, weights
// not in L2): the TMA kernel wins wherever every SM gets a tile (14336 x 4096:
// 12.7-20 us against 24-25 us at M = 2..8; the 128256-row matrix: 58-91 us
// against 179-185 us) and, for M <= 4, down to 64 tiles (4096 x 14336 at M = 2:
// 17 us against 23 us; at M = 4: 22.6 us against 27.4 us, while at M = 6 and 8 the
// general kernel leads, 28 against 33-35 us); with fewer tiles or more rows the general kernel's
// shorter start wins (4096 x 4096 at M = 8: 8.0 us against 12.8 us; 1024 x
// 4096 at M = 2: 5.7 us against 6.2 us).  One row always takes the TMA kernel.
bool qmv_tma_preferred(const MatmulArgs &a) {
    if (a.M == 1) return true;
    // 9..16 rows: where x fits one pass.  In K passes every pass of every tile
    // deposits the partial sums of 16 rows through one buffer (x of 16 rows at
    // K = 4096 is 128 KB): 128256 x 4096 took 204 us, 4096 x 14336 82 us, against
    // 110 us as one launch whose CTA pairs split the rows (taken over at least
    // two tiles per SM) and 28 us on the general kernel.
    if (a.M > kMaxM) return qmv_tma_passes(a) == 1;
    int dev = 0, sms = 0;
    if (device_sms(&dev, &sms) != cudaSuccess) return true;
    const int T = (int)((a.N + kRows - 1) / kRows);
    return T >= sms || (a.M <= 4 && T >= 64);
}

cudaError_t launch_qmv_tma(const MatmulArgs &a) {
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess) return e;
    // M: rows of x per CTA (half of them, rounded up, when CTA pairs split the rows)
    const int M = a.split_rows ? (int)((a.M + 1) / 2) : (int)a.M, N = (int)a.N, K = (int)a.K;
    const int SC = stage_codes(a.bits);
    const int kbp = stages_per_pass(M, K, a.bits);
    const int P = ((K + SC - 1) / SC + kbp - 1) / kbp;
    const bool ns3 = ring_stages(M, K, a.bits) == 3;
    const int T = (N + kRows - 1) / kRows;
    // persistent, one CTA per SM (CTA pairs with split rows: as many pairs as fit)
    const int walkers = a.split_rows ? std::min(T, sms / 2) : std::min(T, sms);
    if (walkers < 1) return cudaErrorInvalidConfiguration;
    const int grid = a.split_rows ? 2 * walkers : walkers;
    const int tpc = (T + walkers - 1) / walkers;
    int cap = 0;   // tiles per batch whose sums stay in shared memory across the passes
    if (P > 1) {
        const int free_bytes = kSmemLimit - 1024 - make_layout(M, kbp * SC, 0, a.bits, ns3 ? 3 : kMaxStages).total;
        cap = std::min(tpc, free_bytes / (kRows * M * 4));
        if (cap < 1) return cudaErrorInvalidConfiguration;
    }
    const Layout L = make_layout(M, P > 1 ? kbp * SC : K, cap, a.bits, ns3 ? 3 : kMaxStages);
    const int smem = L.total + 1024;
    if (smem > kSmemLimit) return cudaErrorInvalidConfiguration;
    const bool one = (M == 1), eight = (a.bits == 8), multi = (P > 1), wide = (M > kMaxM);
    decltype(&qmv_tma_kernel<4, true, false>) kern;
    if (wide)
        kern = eight ? (multi ? (ns3 ? qmv_tma_kernel<8, false, true, 3, 2> : qmv_tma_kernel<8, false, true, 4, 2>)
                              : (ns3 ? qmv_tma_kernel<8, false, false, 3, 2> : qmv_tma_kernel<8, false, false, 4, 2>))
                     : (multi ? (ns3 ? qmv_tma_kernel<4, false, true, 3, 2> : qmv_tma_kernel<4, false, true, 4, 2>)
                              : (ns3 ? qmv_tma_kernel<4, false, false, 3, 2> : qmv_tma_kernel<4, false, false, 4, 2>));
    else if (ns3 && multi)
        kern = eight ? (one ? qmv_tma_kernel<8, true, true, 3> : qmv_tma_kernel<8, false, true, 3>)
                     : (one ? qmv_tma_kernel<4, true, true, 3> : qmv_tma_kernel<4, false, true, 3>);
    else if (ns3)
        kern = eight ? (one ? qmv_tma_kernel<8, true, false, 3> : qmv_tma_kernel<8, false, false, 3>)
                     : (one ? qmv_tma_kernel<4, true, false, 3> : qmv_tma_kernel<4, false, false, 3>);
    else if (multi)
        kern = eight ? (one ? qmv_tma_kernel<8, true, true> : qmv_tma_kernel<8, false, true>)
                     : (one ? qmv_tma_kernel<4, true, true> : qmv_tma_kernel<4, false, true>);
    else
        kern = eight ? (one ? qmv_tma_kernel<8, true, false> : qmv_tma_kernel<8, false, false>)
                     : (one ? qmv_tma_kernel<4, true, false> : qmv_tma_kernel<4, false, false>);
    const int ki = 16 * (int)wide + 8 * (int)ns3 + 4 * (int)multi + 2 * (int)eight + (int)one;
    if (!g_attr_done[ki][dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return e;
        g_attr_done[ki][dev].store(1, std::memory_order_release);
    }
    CUtensorMap tw, ts, tb;
    const int G = K / 64;
    // codes: one stage (8 chunks x 32 rows x 128 bytes, 128-byte swizzle) per box; scales and biases: one
    // stage's groups x 32 rows (64 bytes and 64-byte swizzle for 4-bit codes,
    // 32 bytes and 32-byte swizzle for 8-bit)
    const uint32_t sg = (uint32_t)stage_groups(a.bits);
    const CUtensorMapSwizzle sbs = eight ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!encode_codes_3d(&tw, a.w, (uint64_t)K * a.bits / 8, (uint64_t)N) ||
        !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, (uint64_t)G, (uint64_t)N, (uint64_t)G * 2, sg, kRows,
                   sbs) ||
        !encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.biases, (uint64_t)G, (uint64_t)N, (uint64_t)G * 2, sg, kRows,
                   sbs))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tw, ts, tb, static_cast<const __nv_bfloat16 *>(a.x),
                              static_cast<__nv_bfloat16 *>(a.y), (int)a.M, N, K, kbp, std::max(cap, 1),
                              (unsigned long long)a.timeout_ns,
                              a.status, a.debug_skip_copy ? 1 : 0, a.split_rows ? 1 : 0);
}

}  // namespace aq
