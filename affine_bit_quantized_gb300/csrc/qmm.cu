// Tensor-core kernel for y = x . dequant(W)^T at prefill sizes (M > 16),
// on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// The pages name a quantized GEMM for Blackwell prefill as the large-M
// counterpart of the decode matvec ("epic: CUDA (MLX backend) prefill and
// decode acceleration program", code-audit findings and Phase 6).  At M in
// the hundreds to thousands the work is a real dense contraction, so here it
// runs on tcgen05.mma with fp32 accumulators in tensor memory (TMEM):
//
//   * CTA tile 256 (rows of x; 128 for 8-bit codes unless x is converted once
//     or the CTAs work in pairs) x 256 (rows of W, or 224 where that fills the
//     last wave), K walked one group of 64 at a time; two 128 x 256 fp32
//     accumulators fill the 512 TMEM columns.
//   * warp 0 (one thread) streams raw tiles with TMA: x (bf16, 128-byte
//     swizzle), the packed codes of the 256 W rows, and every 8 groups the
//     rows' bf16 scales and biases;
//   * warps 2..17 turn a raw stage into the MMA operands, in the canonical
//     K-major 128-byte-swizzled layout: W is dequantized to fp16 as
//     fp16(scale * q + bias) (q made exact with the 1024 + q exponent trick,
//     then one HFMA2, so one rounding per weight), and x is converted from
//     bf16 to fp16.  fp16 rather than bf16 because a bf16 weight (8-bit
//     significand) perturbs y by about twice the tolerance on these shapes,
//     while fp16 (11 bits) stays about 6 sigma inside it.  Inside every
//     8-element chunk both operands use the k order (0,4,1,5,2,6,3,7)
//     ((0,2,1,3,4,6,5,7) for 8-bit codes), which lets one LOP3 build a pair
//     of codes; the dot product is unchanged;
//   * with a caller workspace (XPRE) x is converted to fp16 once by a small
//     kernel and the TMA copies it straight into the operand tile: the
//     converters only build W, and the freed raw x stage becomes a third
//     converted stage (the expert-indexed path always works this way);
//   * warp 1 allocates TMEM and one of its threads issues the MMAs
//     (M=128, N=256, K=16, both operands from shared memory), committing each
//     consumed stage back to the converters through an mbarrier;
//   * after the last group, warps 2..9 read the accumulators with tcgen05.ld,
//     round to bf16 and store y; with few output tiles, K is split across a
//     cluster and the partial tiles are added through distributed shared
//     memory first (see the epilogue);
//   * where each CTA converts its own x tiles and K is not split, two CTAs of a
//     cluster share each W tile (tcgen05 cta_group::2, see qmm_kernel).
//
// Every mbarrier wait is bounded by a global-timer deadline; on expiry the
// kernel records a timeout in the device status word, stops issuing work,
// waits (bounded) for what it already issued, frees its TMEM and returns.
//
// Numerics precondition of this path: x, scales and biases inside the fp16
// normal range (|v| < 65504; magnitudes below 2^-14 lose relative precision).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "aq_internal.h"

namespace aq {
namespace {

constexpr int kTileN = 256;            // rows of W per CTA (UMMA N)
constexpr int kGroup = 64;             // K per pipeline step (one quantization group)
constexpr int kConvWarps = 16;
constexpr int kThreads = (2 + kConvWarps) * 32;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kSBGroups = 8;           // groups of scales/biases per TMA box (16 bytes per row)
constexpr int kSBStages = 2;

// Shared-memory layout for a code width (offsets from a 1024-aligned base).
// 4-bit codes: 256 rows of x per CTA (two UMMA M=128 halves); 8-bit codes
// carry twice the raw bytes per W row, and 128 rows of x keep the stages
// within the 227 KB a CTA may use.  XPRE: x arrives already in fp16 (in the
// MMA's k order, from a conversion pass into the caller's workspace), copied
// by TMA straight into the operand tile: no raw x stage, which leaves room
// for a third converted stage.
// TM: rows of x per CTA.  kXInConv: x (fp16 with XPRE; bf16 with 8-bit codes on
// 256-row tiles, which the converters turn into fp16 in place) is copied by TMA
// straight into the x tile of a converted stage, so there is no raw x stage: the
// 8-bit 256-row tiles get four converted stages instead of two (M = 2048 without
// the workspace: 255 -> 202 us).  Otherwise bf16 x comes with the codes in the raw
// stage, two to four stages ahead of the converters, and is converted into the converted
// stage: in the converted stage the copy's latency would sit on the loop from the
// MMAs back to the converters (4-bit M = 2048 on 14336 x 4096: 186 -> 196 us; 8-bit
// 128-row pairs at M = 256: 58 -> 65 us).  As many converted stages as fit (at
// most 4) follow the raw and scale/bias stages.
// PAIR (without XPRE): the CTA holds half of the W tile (see qmm_kernel).
// TN: rows of W the stages are laid out for (kTileN, or 224: smaller stages, more of them).
template <int BITS, bool XPRE = false, int TM = (BITS == 4 ? 256 : 128), bool PAIR = false, int TN = kTileN>
struct Cfg {
    static constexpr int kTileM = TM;
    static constexpr int kHalves = kTileM / 128;                 // UMMA M=128 accumulators
    static constexpr int kWRows = PAIR ? TN / 2 : TN;           // rows of W in this CTA's stages
    static constexpr int kBTileBytes = kWRows * 128;             // fp16 W, kWRows rows x 64 k
    static constexpr int kSBBytes = kWRows * kSBGroups * 2;      // scales (and again biases) per stage
    static constexpr bool kXInConv = XPRE || (BITS == 8 && TM == 256);
    static constexpr int kATileBytes = kTileM * 128;             // x, kTileM rows x 64 k (fp16 once converted)
    static constexpr int kConvStageBytes = kATileBytes + kBTileBytes;
    static constexpr int kRawXBytes = kXInConv ? 0 : kTileM * 128;   // bf16 x, same swizzled geometry
    static constexpr int kRowWords = kGroup * BITS / 32;         // code words per W row and group
    static constexpr int kRawCodeBytes = kWRows * kRowWords * 4; // 8192 or 16384 (half in a pair)
    static constexpr int kRawStageBytes = kRawXBytes + kRawCodeBytes;
    // converted stages (at most 4) that fit beside R raw stages, the scale/bias stages, room for
    // the barriers and the alignment slack
    static constexpr int conv_fit(int R) {
        return (232448 - (R * kRawStageBytes + kSBStages * 2 * kSBBytes + 512 + 16 + 1024)) / kConvStageBytes < 4
                   ? (232448 - (R * kRawStageBytes + kSBStages * 2 * kSBBytes + 512 + 16 + 1024)) / kConvStageBytes
                   : 4;
    }
    // Raw stages: each raw stage's loop is the copy's latency plus its conversion, so the ring's
    // depth bounds the step rate wherever a step carries little work.  128-row tiles of one CTA
    // (prefill at M = 256, where the K split leaves each CTA few steps) take 4 raw stages (3 for
    // 8-bit codes with bf16 x) even where that leaves two converted stages; CTA pairs deepen the
    // ring (up to 4) only where the converted stages keep their number.  Measured at M = 256:
    // 4-bit 60.0 -> 58.6 us (59.3 -> 55.6 with x converted once), 8-bit 64.4 -> 59.9 us and
    // 55.6 -> 48.3 us; 8-bit 256-row pairs at M = 2048: 204.6 -> 194.8 us.  256-row tiles of
    // one CTA keep two (8-bit with x converted once measured 0.6 % slower with four).
    static constexpr int kRawStages =
        (TM == 128 && !PAIR) ? (conv_fit(4) >= 2 ? 4 : 3)
        : PAIR ? (conv_fit(4) == conv_fit(2) ? 4 : conv_fit(3) == conv_fit(2) ? 3 : 2)
               : 2;
    static constexpr int kConvStages = conv_fit(kRawStages);
    // barriers: raw_full[R], raw_empty[R], sb_full[2], sb_empty[2], conv_full[S], conv_empty[S], acc_done,
    // x_full[S] (the x copy of a converted stage has landed) and peer_full[S] (in a CTA pair: the
    // other CTA's half of a converted stage is ready)
    static constexpr int kNumBars = 2 * kRawStages + 2 * kSBStages + 4 * kConvStages + 1;
    static constexpr int kOffConv = 0;
    static constexpr int kOffRaw = kOffConv + kConvStages * kConvStageBytes;
    static constexpr int kOffSB = kOffRaw + kRawStages * kRawStageBytes;
    static constexpr int kOffBar = kOffSB + kSBStages * 2 * kSBBytes;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;     // tmem address, abort flag
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;     // + alignment slack
};
static_assert(Cfg<4>::kSmemBytes <= 232448 && Cfg<8>::kSmemBytes <= 232448 && Cfg<4, true>::kSmemBytes <= 232448 &&
                  Cfg<8, true>::kSmemBytes <= 232448 && Cfg<8, true, 256>::kSmemBytes <= 232448 &&
                  Cfg<4, false, 256, true>::kSmemBytes <= 232448 && Cfg<8, false, 128, true>::kSmemBytes <= 232448 &&
                  Cfg<8, false, 256, true>::kSmemBytes <= 232448 && Cfg<4, false, 128>::kSmemBytes <= 232448 &&
                  Cfg<8, true, 256, false, 224>::kSmemBytes <= 232448 &&
                  Cfg<4, true, 128>::kSmemBytes <= 232448 && Cfg<4>::kConvStages >= 2 && Cfg<8>::kConvStages >= 2 &&
                  Cfg<8, true, 256>::kConvStages >= 2,
              "shared memory per CTA");
// split-K partials received by a CTA (at most 7 sources x its 32 columns x the tile's rows) fit in
// the stage memory in front of the barriers
constexpr int kMaxSplit = 8;
static_assert((kMaxSplit - 1) * Cfg<4>::kTileM * (kTileN / kMaxSplit) * 4 <= Cfg<4>::kOffBar &&
                  (kMaxSplit - 1) * Cfg<8>::kTileM * (kTileN / kMaxSplit) * 4 <= Cfg<8>::kOffBar &&
                  (kMaxSplit - 1) * Cfg<4, true>::kTileM * (kTileN / kMaxSplit) * 4 <= Cfg<4, true>::kOffBar &&
                  (kMaxSplit - 1) * Cfg<8, true>::kTileM * (kTileN / kMaxSplit) * 4 <= Cfg<8, true>::kOffBar &&
                  (kMaxSplit - 1) * Cfg<4, false, 128>::kTileM * (kTileN / kMaxSplit) * 4 <= Cfg<4, false, 128>::kOffBar &&
                  (kMaxSplit - 1) * Cfg<4, true, 128>::kTileM * (kTileN / kMaxSplit) * 4 <= Cfg<4, true, 128>::kOffBar,
              "split-K receive slots");
// 256-row 8-bit tiles are taken only without a split

constexpr uint32_t kTmemCols = 512;
constexpr int kPlanHeaderInts = 32;    // tile count, then the tiles (int4 each) from byte 128

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// the abort flag and the timer are looked at every 16th poll, so that a completed
// phase is seen a few cycles sooner
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t deadline,
                                          const volatile int *abort_flag) {
    for (uint32_t n = 0; !mbar_try_wait(bar, parity); ++n) {
        if ((n & 15) != 15) continue;
        if (*abort_flag) return false;
        if (global_timer() > deadline) return false;
    }
    return true;
}
// the same wait at cluster scope: the arrivals come from the other CTA of a pair
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t deadline,
                                                  const volatile int *abort_flag) {
    for (uint32_t n = 0; !mbar_try_wait_cluster(bar, parity); ++n) {
        if ((n & 15) != 15) continue;
        if (*abort_flag) return false;
        if (global_timer() > deadline) return false;
    }
    return true;
}
// arrive on an mbarrier of another CTA of the cluster (its shared::cluster address)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// fp16x2 (1024 + q[p], 1024 + q[p+4]) from a word shifted right by 4p.
__device__ __forceinline__ uint32_t code_pair_f16(uint32_t v, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(r) : "r"(v), "r"(magic));
    return r;
}
// Eight bf16 x values (one 16-byte chunk) as fp16 in the MMA's k order within the
// chunk: (0,4,1,5,2,6,3,7) for 4-bit codes, (0,2,1,3,4,6,5,7) for 8-bit codes --
// the order the code pairs of W come in.
template <int BITS>
__device__ __forceinline__ uint4 x_chunk_f16(uint4 v);

// fp16x2 (1024 + byte 0, 1024 + byte 2) of a word: exact for bytes up to 255.
__device__ __forceinline__ uint32_t byte_pair_f16(uint32_t v, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, 0x00FF00FF, %2, 0xEA;" : "=r"(r) : "r"(v), "r"(magic));
    return r;
}
// fp16x2: (pair - 1024) * s + b, with the subtraction exact and one rounding in the FMA
__device__ __forceinline__ uint32_t dequant_pair(uint32_t pair, uint32_t s2, uint32_t b2, uint32_t off2) {
    uint32_t q, w;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(q) : "r"(pair), "r"(off2));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(w) : "r"(q), "r"(s2), "r"(b2));
    return w;
}
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(uint32_t lo, uint32_t hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    return r;
}
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
    d |= (uint64_t)1 << 16;                   // leading-dimension offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;         // stride-dimension offset: next 8-row group
    d |= (uint64_t)1 << 46;                   // descriptor version
    d |= (uint64_t)2 << 61;                   // 128-byte swizzle
    return d;
}
// instruction descriptor: D f32, A f16, B f16, both K-major, M (128, or 256 over a CTA pair),
// N=tn (256 or 224)
__host__ __device__ constexpr uint32_t umma_idesc(int tn, int m = 128) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(tn >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// CTA pair (cta_group::2): one MMA of M = 256 rows of x, 128 from each CTA's A tile, over
// N rows of W of which each CTA holds N/2 in its B tile (the first half in the even CTA);
// each CTA's accumulators hold its own 128 rows.  Issued by the even CTA only.
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on the mbarrier at this offset in both CTAs of the pair once the MMAs issued so far are done
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"((uint16_t)3)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// all threads of every CTA of the cluster; release/acquire orders shared::cluster memory
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_cta(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int BITS>
__device__ __forceinline__ uint4 x_chunk_f16(uint4 v) {
    uint4 o;
    if (BITS == 4) {
        o.x = f32x2_to_f16x2(bf16lo(v.x), bf16lo(v.z));
        o.y = f32x2_to_f16x2(bf16hi(v.x), bf16hi(v.z));
        o.z = f32x2_to_f16x2(bf16lo(v.y), bf16lo(v.w));
        o.w = f32x2_to_f16x2(bf16hi(v.y), bf16hi(v.w));
    } else {
        o.x = f32x2_to_f16x2(bf16lo(v.x), bf16lo(v.y));
        o.y = f32x2_to_f16x2(bf16hi(v.x), bf16hi(v.y));
        o.z = f32x2_to_f16x2(bf16lo(v.z), bf16lo(v.w));
        o.w = f32x2_to_f16x2(bf16hi(v.z), bf16hi(v.w));
    }
    return o;
}

// x [rows][K] bf16 -> fp16 in the MMA's chunk order (x_chunk_f16), 16 bytes per
// thread and step: the conversion every CTA of the tensor-core kernel would
// otherwise repeat on its raw x tiles.
template <int BITS>
__global__ void x_to_f16_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ xf, int64_t vecs) {
    griddep_launch();   // the tensor-core kernel after it may start its set-up (it waits for xf)
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs; i += (int64_t)gridDim.x * blockDim.x)
        xf[i] = x_chunk_f16<BITS>(__ldg(x + i));
}

// A plain launch whose error comes back from the call itself (not through
// cudaGetLastError, which would also report an earlier, unrelated failure).
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// GROUPED (expert-indexed matmul): x holds the rows gathered in expert order,
// W, scales and biases are E matrices stacked along N, and `plan` lists the
// work tiles {expert, first row, rows} (see gather_plan_kernel); CTA row
// blockIdx.y takes tile blockIdx.y and exits at once if there is none.
// Plain matmul, order of the tiles (mfast): where W is the larger operand, row
// tiles of x run fastest (blockIdx.x: row tile of x, blockIdx.y: tile of W), so
// that a wave of CTAs finishes a band of W tiles (each read from DRAM once) while
// x stays in L2; otherwise W tiles run fastest (blockIdx.x: tile of W).
// PAIR: a cluster of two CTAs, along the cluster's x (row tiles 2j and 2j + 1 of
// x: blockIdx.x = 2j + rank with mfast, else blockIdx.x = 2 (W tile) + rank and
// blockIdx.y = j), shares one tile of tn rows of W: each CTA loads and converts tn/2 of them (the even CTA the
// first half) and its own TM rows of x, and the even CTA issues the MMAs for
// both (tcgen05 cta_group::2, M = 256 across the pair), so every W element is
// converted, stored and read from shared memory once per 2 TM rows of x.  Only
// without a K split, and only where each CTA converts its own x tiles: there the
// converters bound the step and the pair takes a quarter of their work away
// (M = 2048 on 4096 x 14336: 214 -> 201 us); with x converted once the MMAs
// bound it and the pair's MMAs ran slower than two single-CTA ones.
template <int BITS, bool GROUPED, bool XPRE, int TM = (BITS == 4 ? 256 : 128), bool PAIR = false, int TN = kTileN>
__global__ void __launch_bounds__(kThreads, 1)
qmm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
           const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_b,
           __nv_bfloat16 *__restrict__ y, int M, int N, int K, unsigned long long timeout_ns, int *status,
           const int *__restrict__ plan, int skip_copy, int tn, int mfast, int tile0) {
    static_assert(!(PAIR && (GROUPED || XPRE)), "CTA pairs only on the plain matmul without x converted once");
    using C = Cfg<BITS, XPRE, TM, PAIR, TN>;
    constexpr int kSBBytes = C::kSBBytes;
    constexpr int kConvStages = C::kConvStages, kRawStages = C::kRawStages;
    constexpr int kTileM = C::kTileM, kATileBytes = C::kATileBytes, kConvStageBytes = C::kConvStageBytes;
    constexpr int kRawXBytes = C::kRawXBytes, kRawStageBytes = C::kRawStageBytes;
    constexpr bool kXInConv = C::kXInConv;
    constexpr int kOffConv = C::kOffConv, kOffRaw = C::kOffRaw, kOffSB = C::kOffSB, kOffMisc = C::kOffMisc;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_base);

    const uint32_t bar0 = base + C::kOffBar;
    auto raw_full = [&](int s) { return bar0 + 8 * s; };
    auto raw_empty = [&](int s) { return bar0 + 8 * (kRawStages + s); };
    auto sb_full = [&](int s) { return bar0 + 8 * (2 * kRawStages + s); };
    auto sb_empty = [&](int s) { return bar0 + 8 * (2 * kRawStages + kSBStages + s); };
    auto conv_full = [&](int s) { return bar0 + 8 * (2 * kRawStages + 2 * kSBStages + s); };
    auto conv_empty = [&](int s) { return bar0 + 8 * (2 * kRawStages + 2 * kSBStages + kConvStages + s); };
    const uint32_t acc_done = bar0 + 8 * (2 * kRawStages + 2 * kSBStages + 2 * kConvStages);
    auto x_full = [&](int s) { return acc_done + 8 * (1 + s); };
    auto peer_full = [&](int s) { return acc_done + 8 * (1 + kConvStages + s); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // tn: rows of W per output tile (per CTA, or per CTA pair), kTileN or 224 (a full
    // last wave where 256 would leave SMs idle; only without a K split); the stage
    // memory is laid out for kTileN.  prank: rank in the CTA pair (0 issues the MMAs).
    const uint32_t prank = PAIR ? cluster_rank() : 0u;
    const int bx = (int)blockIdx.x, by = (int)blockIdx.y;
    const int n0 = (GROUPED ? bx : mfast ? by : PAIR ? bx >> 1 : bx) * tn;
    int m0 = (GROUPED ? 0 : mfast ? bx : PAIR ? 2 * by + (int)prank : by) * kTileM;   // first row of x (and y)
    int m_end = M;                  // rows from m_end on are not this tile's
    const int wrows = PAIR ? tn / 2 : tn;   // rows of W this CTA loads and converts
    int wrow0 = n0 + (int)prank * wrows;    // the first of them (in the stacked experts: expert * N + ...)
    int halves = C::kHalves;                 // M=128 accumulators in use
    if (GROUPED) {
        const int ti = (int)blockIdx.y + tile0;   // this launch's tiles start at the plan's tile0
        if (ti >= __ldg(plan)) return;              // no tile: nothing set up yet
        const int4 t = __ldg(reinterpret_cast<const int4 *>(plan + kPlanHeaderInts) + ti);
        m0 = t.y;
        m_end = t.y + t.z;
        wrow0 = t.x * N + n0;
        // an expert's last tile with at most 128 rows (the few rows past a multiple of 256)
        // runs only the first half's MMAs and epilogue: half the operand reads per step
        if (t.z <= 128) halves = 1;
    }
    // split K: the gridDim.z CTAs of a cluster each take a contiguous share of
    // the K/512 blocks of 8 groups and add their partial tiles through
    // distributed shared memory at the end
    const int nsplit = (int)gridDim.z, split = (int)blockIdx.z;
    const int blocks = K / (kGroup * kSBGroups);
    const int blk0 = split * blocks / nsplit, blk1 = (split + 1) * blocks / nsplit;
    const int g0 = blk0 * kSBGroups;                // first group of this CTA
    const int steps = (blk1 - blk0) * kSBGroups;    // groups of this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(raw_full(s), 1);
            mbar_init(raw_empty(s), kConvWarps);
        }
        for (int s = 0; s < kSBStages; ++s) {
            mbar_init(sb_full(s), 1);
            mbar_init(sb_empty(s), kConvWarps);
        }
        for (int s = 0; s < kConvStages; ++s) {
            mbar_init(x_full(s), 1);
            if (PAIR) mbar_init(peer_full(s), 1);
            mbar_init(conv_full(s), kConvWarps);
            mbar_init(conv_empty(s), 1);
        }
        mbar_init(acc_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            // one warp of each CTA of the pair, together: the same columns in both
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_addr(tmem_slot)),
                         "r"(kTmemCols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_addr(tmem_slot)),
                         "r"(kTmemCols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    if (PAIR)
        cluster_sync();   // both CTAs' barriers initialised before either signals the other
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_launch();
    griddep_wait();  // x (and y) may belong to the preceding kernel
    const uint64_t deadline = global_timer() + timeout_ns;

    auto fail = [&]() {
        if (!*abort_flag) {
            atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
            *abort_flag = 1;
        }
    };
    // epilogue geometry of warps 2..kEpiEnd-1: TMEM lane quarter q, accumulator half h
    // (x rows 128h..128h+127), this lane's row m of y
    constexpr int kEpiEnd = 2 + 4 * C::kHalves;
    const int q = warp & 3;
    const int h = warp >= 2 ? (warp - 2) >> 2 : 0;
    const int m = m0 + h * 128 + q * 32 + lane;
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * kTileN);
    bool go = false;   // this warp holds final accumulators to write out
    // 16 fp32 values of row m, columns n..n+15 -> bf16 y
    auto store_row16 = [&](const float (&a)[16], int m_, int n) {
        if (m_ >= m_end) return;
        __nv_bfloat16 *yp = y + (int64_t)m_ * N + n;
        if (n + 16 <= N && (((uintptr_t)yp) & 15) == 0) {
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                uint4 o;
                o.x = f32x2_to_bf16x2(__float_as_uint(a[8 * v + 0]), __float_as_uint(a[8 * v + 1]));
                o.y = f32x2_to_bf16x2(__float_as_uint(a[8 * v + 2]), __float_as_uint(a[8 * v + 3]));
                o.z = f32x2_to_bf16x2(__float_as_uint(a[8 * v + 4]), __float_as_uint(a[8 * v + 5]));
                o.w = f32x2_to_bf16x2(__float_as_uint(a[8 * v + 6]), __float_as_uint(a[8 * v + 7]));
                *reinterpret_cast<uint4 *>(yp + 8 * v) = o;
            }
        } else {
#pragma unroll
            for (int v = 0; v < 16; ++v)
                if (n + v < N) yp[v] = __float2bfloat16_rn(a[v]);
        }
    };
    // 32 fp32 values of row m, columns n..n+31 -> bf16 y
    auto store_row32 = [&](const uint32_t (&r)[32], int m_, int n) {
        if (m_ >= m_end) return;
        __nv_bfloat16 *yp = y + (int64_t)m_ * N + n;
        if (n + 32 <= N && (((uintptr_t)yp) & 15) == 0) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = f32x2_to_bf16x2(r[8 * v + 0], r[8 * v + 1]);
                o.y = f32x2_to_bf16x2(r[8 * v + 2], r[8 * v + 3]);
                o.z = f32x2_to_bf16x2(r[8 * v + 4], r[8 * v + 5]);
                o.w = f32x2_to_bf16x2(r[8 * v + 6], r[8 * v + 7]);
                *reinterpret_cast<uint4 *>(yp + 8 * v) = o;
            }
        } else {
#pragma unroll
            for (int v = 0; v < 32; ++v)
                if (n + v < N) yp[v] = __float2bfloat16_rn(__uint_as_float(r[v]));
        }
    };

    int issued_raw = 0, issued_sb = 0, issued_conv = 0;   // copies issued (producer thread)
    // let every copy issued land before the CTA may exit (bounded)
    auto drain_copies = [&]() {
        const uint64_t drain = global_timer() + timeout_ns;
        for (int i = (issued_raw > kRawStages ? issued_raw - kRawStages : 0); i < issued_raw; ++i)
            while (!mbar_try_wait(raw_full(i % kRawStages), (i / kRawStages) & 1) && global_timer() < drain) {
            }
        for (int j = (issued_sb > kSBStages ? issued_sb - kSBStages : 0); j < issued_sb; ++j)
            while (!mbar_try_wait(sb_full(j % kSBStages), (j / kSBStages) & 1) && global_timer() < drain) {
            }
        if (kXInConv)
            for (int i = (issued_conv > kConvStages ? issued_conv - kConvStages : 0); i < issued_conv; ++i)
                while (!mbar_try_wait(x_full(i % kConvStages), (i / kConvStages) & 1) && global_timer() < drain) {
                }
    };
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // test hook: the first CTA leaves out its first raw copy, so its consumers' wait expires
            const bool skip_first = skip_copy && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
            bool ok = true;
            for (int i = 0; i < steps && ok; ++i) {
                const int rs = i % kRawStages;
                if (i % kSBGroups == 0) {
                    const int j = i / kSBGroups, ss = j % kSBStages;
                    if (j >= kSBStages && !mbar_wait(sb_empty(ss), ((j / kSBStages) - 1) & 1, deadline, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + kOffSB + ss * 2 * kSBBytes;
                    mbar_expect_tx(sb_full(ss), (uint32_t)(2 * wrows * kSBGroups * 2));
                    tma_load_2d(dst, &tm_s, g0 + j * kSBGroups, wrow0, sb_full(ss));
                    tma_load_2d(dst + kSBBytes, &tm_b, g0 + j * kSBGroups, wrow0, sb_full(ss));
                    issued_sb = j + 1;
                }
                if (i >= kRawStages && !mbar_wait(raw_empty(rs), ((i / kRawStages) - 1) & 1, deadline, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = base + kOffRaw + rs * kRawStageBytes;
                if (!(skip_first && i == 0)) {
                    mbar_expect_tx(raw_full(rs), (uint32_t)(kRawXBytes + wrows * C::kRowWords * 4));
                    if (!kXInConv) tma_load_2d(dst, &tm_x, (g0 + i) * kGroup, m0, raw_full(rs));
                    tma_load_2d(dst + kRawXBytes, &tm_w, (g0 + i) * C::kRowWords, wrow0, raw_full(rs));
                }
                issued_raw = i + 1;
                if (kXInConv) {
                    // x straight into the converted stage, once the MMAs have released it
                    const int cs = i % kConvStages;
                    if (i >= kConvStages &&
                        !mbar_wait(conv_empty(cs), ((i / kConvStages) - 1) & 1, deadline, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(x_full(cs), kATileBytes);
                    tma_load_2d(base + kOffConv + cs * kConvStageBytes, &tm_x, (g0 + i) * kGroup, m0, x_full(cs));
                    issued_conv = i + 1;
                }
            }
            if (!ok) fail();   // the copies issued are drained at the end of the kernel
        }
    } else if (warp == 1 && PAIR && prank != 0) {
        // ------------------------------------------------------------ pair: stage readiness to the MMA CTA
        if (lane == 0) {
            for (int i = 0; i < steps; ++i) {
                const int cs = i % kConvStages;
                if (!mbar_wait(conv_full(cs), (i / kConvStages) & 1, deadline, abort_flag)) {
                    fail();
                    break;
                }
                mbar_arrive_cluster(map_cta(peer_full(cs), 0));
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc(tn, PAIR ? 256 : 128);
            for (int i = 0; i < steps; ++i) {
                const int cs = i % kConvStages;
                if (!mbar_wait(conv_full(cs), (i / kConvStages) & 1, deadline, abort_flag) ||
                    (XPRE && !mbar_wait(x_full(cs), (i / kConvStages) & 1, deadline, abort_flag)) ||
                    (PAIR && !mbar_wait_cluster(peer_full(cs), (i / kConvStages) & 1, deadline, abort_flag))) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = base + kOffConv + cs * kConvStageBytes;
                const uint32_t b0 = a0 + kATileBytes;
#pragma unroll
                for (int kk = 0; kk < kGroup / 16; ++kk) {
                    const uint64_t bd = sw128_desc(b0 + kk * 32);
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h) {
                        if (h >= halves) break;
                        if constexpr (PAIR)
                            umma_f16_pair(tmem + h * kTileN, sw128_desc(a0 + h * (128 * 128) + kk * 32), bd, idesc,
                                          (i > 0 || kk > 0) ? 1u : 0u);
                        else
                            umma_f16(tmem + h * kTileN, sw128_desc(a0 + h * (128 * 128) + kk * 32), bd, idesc,
                                     (i > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                if constexpr (PAIR)
                    umma_commit_pair(conv_empty(cs));
                else
                    umma_commit(conv_empty(cs));
            }
            // acc_done fires when every MMA issued so far has completed (also on abort)
            if constexpr (PAIR)
                umma_commit_pair(acc_done);
            else
                umma_commit(acc_done);
        }
    } else {
        // ------------------------------------------------------------ converters
        const int t = threadIdx.x - 64;  // 0..kConvThreads-1
        const uint32_t magic = 0x64006400u;   // fp16x2 (1024, 1024)
        const uint32_t off2 = 0x64006400u;
        bool alive = true;
        for (int i = 0; i < steps; ++i) {
            const int rs = i % kRawStages, cs = i % kConvStages, ss = (i / kSBGroups) % kSBStages;
            if (alive && !mbar_wait(raw_full(rs), (i / kRawStages) & 1, deadline, abort_flag)) alive = false;
            if (alive && !mbar_wait(sb_full(ss), (i / (kSBGroups * kSBStages)) & 1, deadline, abort_flag))
                alive = false;
            if (alive && i >= kConvStages &&
                !mbar_wait(conv_empty(cs), ((i / kConvStages) - 1) & 1, deadline, abort_flag))
                alive = false;
            alive = __all_sync(0xFFFFFFFFu, alive);  // keep the warp's decisions uniform
            if (!alive) {
                fail();
                break;
            }
            const uint32_t raw = base + kOffRaw + rs * kRawStageBytes;
            const uint32_t conv = base + kOffConv + cs * kConvStageBytes;
            if (!kXInConv) {
                // x: bf16 -> fp16 from the raw stage, chunk by chunk at the same (swizzled) offsets,
                // each chunk's k order becoming (0,4,1,5,2,6,3,7) (the order the W pairs come in)
#pragma unroll 4
                for (int c = 0; c < kRawXBytes / 16 / kConvThreads; ++c) {
                    const uint32_t off = (uint32_t)((c * kConvThreads + t) * 16);
                    sts128(conv + off, x_chunk_f16<BITS>(lds128(raw + off)));
                }
            }
            // W: thread t takes chunks kCpt*p .. kCpt*p + kCpt-1 of row r = t / kTpr
            // (p = t % kTpr) and converts the row's scale and bias once; each chunk of
            // 8 codes becomes 8 fp16 weights at row r, chunk c ^ (r & 7)
            const uint32_t sb = base + kOffSB + ss * 2 * kSBBytes;
            const int g8 = i % kSBGroups;
            constexpr int kTpr = PAIR ? 4 : 2, kCpt = 8 / kTpr;   // threads per row, chunks per thread
            static_assert(kConvThreads == kTpr * (PAIR ? kTileN / 2 : kTileN), "converter threads per W row");
            if (t / kTpr < wrows) {   // rows past wrows are not loaded and not used
                const int r = t / kTpr, hw = t % kTpr;
                const __half sh = __float2half_rn(__uint_as_float((uint32_t)lds16(sb + (r * kSBGroups + g8) * 2) << 16));
                const __half bh =
                    __float2half_rn(__uint_as_float((uint32_t)lds16(sb + kSBBytes + (r * kSBGroups + g8) * 2) << 16));
                const uint32_t s2 = (uint32_t)__half_as_ushort(sh) * 0x00010001u;
                const uint32_t b2 = (uint32_t)__half_as_ushort(bh) * 0x00010001u;
                const uint32_t wrow = raw + kRawXBytes + r * (C::kRowWords * 4) + hw * (C::kRowWords * 4 / kTpr);
                if (BITS == 4) {
                    // word c of the row holds chunk c: pairs (p, p+4) from the word shifted by 4p
                    uint32_t wvs[kCpt];
                    if constexpr (kCpt == 4) {
                        const uint4 v = lds128(wrow);
                        wvs[0] = v.x, wvs[1] = v.y, wvs[2] = v.z, wvs[3] = v.w;
                    } else {
                        const uint2 v = lds64(wrow);
                        wvs[0] = v.x, wvs[1] = v.y;
                    }
#pragma unroll
                    for (int e = 0; e < kCpt; ++e) {
                        const uint32_t w = wvs[e];
                        const int c = kCpt * hw + e;
                        uint4 o;
                        o.x = dequant_pair(code_pair_f16(w, magic), s2, b2, off2);
                        o.y = dequant_pair(code_pair_f16(w >> 4, magic), s2, b2, off2);
                        o.z = dequant_pair(code_pair_f16(w >> 8, magic), s2, b2, off2);
                        o.w = dequant_pair(code_pair_f16(w >> 12, magic), s2, b2, off2);
                        sts128(conv + kATileBytes + r * 128 + ((c ^ (r & 7)) << 4), o);
                    }
                } else {
                    // words 2c, 2c+1 hold chunk c: bytes (0,2) and (1,3) of each word pair up
#pragma unroll
                    for (int hh = 0; hh < kCpt / 2; ++hh) {
                        const uint4 wv = lds128(wrow + hh * 16);
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint32_t wa = e == 0 ? wv.x : wv.z, wb = e == 0 ? wv.y : wv.w;
                            const int c = kCpt * hw + 2 * hh + e;
                            uint4 o;
                            o.x = dequant_pair(byte_pair_f16(wa, magic), s2, b2, off2);
                            o.y = dequant_pair(byte_pair_f16(wa >> 8, magic), s2, b2, off2);
                            o.z = dequant_pair(byte_pair_f16(wb, magic), s2, b2, off2);
                            o.w = dequant_pair(byte_pair_f16(wb >> 8, magic), s2, b2, off2);
                            sts128(conv + kATileBytes + r * 128 + ((c ^ (r & 7)) << 4), o);
                        }
                    }
                }
            }
            if (kXInConv && !XPRE) {
                // x: the bf16 copy in the stage's x tile becomes fp16 in place, chunk by chunk
                // at the same (swizzled) offsets, each chunk's k order becoming (0,2,1,3,4,6,5,7)
                // (the order the 8-bit W pairs come in; only 8-bit codes take this way); W above
                // did not need it, so its conversion overlapped the copy
                bool xok = mbar_wait(x_full(cs), (i / kConvStages) & 1, deadline, abort_flag);
                xok = __all_sync(0xFFFFFFFFu, xok);
                if (!xok) {
                    alive = false;
                    fail();
                    break;
                }
                // the TMA wrote the tile (async proxy); these generic loads follow its completion
#pragma unroll 4
                for (int c = 0; c < kATileBytes / 16 / kConvThreads; ++c) {
                    const uint32_t off = (uint32_t)((c * kConvThreads + t) * 16);
                    sts128(conv + off, x_chunk_f16<BITS>(lds128(conv + off)));
                }
            }
            fence_proxy_async();  // make the generic-proxy stores visible to the MMA (async proxy)
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(conv_full(cs));
                mbar_arrive(raw_empty(rs));
                if (g8 == kSBGroups - 1 || i == steps - 1) mbar_arrive(sb_empty(ss));
            }
        }
        // ------------------------------------------------------------ epilogue
        // warps 2..(1 + 4 x halves) read the accumulators (one per TMEM lane quarter and half)
        const bool epi = warp < kEpiEnd && h < halves;   // this warp's accumulators are in use
        go = epi && alive && mbar_wait(acc_done, 0, deadline, abort_flag) && !*abort_flag;
        go = __all_sync(0xFFFFFFFFu, go);   // tcgen05.ld below is warp-collective
        if (go) {
            tc_fence_after();
            if (nsplit == 1) {
#pragma unroll 1
                for (int j = 0; j < tn / 32; ++j) {
                    uint32_t r[32];
                    tmem_ld32(tbase + j * 32, r);
                    store_row32(r, m, n0 + j * 32);
                }
            }
        } else if (alive && epi) {
            fail();
        }
    }

    if (nsplit > 1) {
        // Split-K sum.  CTA o of the cluster owns columns [o W, (o + 1) W) of the
        // tile (W = 256 / nsplit); every other CTA writes its partial of those
        // columns into o's (now idle) stage memory, and o adds the partials in
        // cluster-rank order (deterministic) and stores y.  Receive slot of
        // source z at owner o: z - (z > o); rows of W floats, 16-byte units
        // XOR-swizzled by row so the stores spread over the banks.
        const int W = kTileN / nsplit;
        const uint32_t me = cluster_rank();
        const uint32_t recv = base + kOffConv;
        auto unit_addr = [&](int slot, int row, int col, int v) {   // col: first column of a 32-column chunk
            return recv + (uint32_t)(((slot * kTileM + row) * W + col) * 4 + (((v ^ (row & 7)) & 7) << 4));
        };
        cluster_sync();   // every partial final, every CTA's stage memory free
        const int row = m - m0;
        if (go) {
#pragma unroll 1
            for (int j = 0; j < kTileN / 32; ++j) {
                const int o = j * 32 / W;
                if (o == (int)me) continue;
                uint32_t r[32];
                tmem_ld32(tbase + j * 32, r);
                const int slot = (int)me - ((int)me > o ? 1 : 0);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    st_cluster128(map_cta(unit_addr(slot, row, j * 32 - o * W, v), (uint32_t)o), r[4 * v],
                                  r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
            }
        }
        cluster_sync();   // every partial delivered
        if (go) {
            // 16 columns at a time: the own partial from TMEM, the others from the receive slots
#pragma unroll 1
            for (int c = (int)me * W; c < ((int)me + 1) * W; c += 16) {
                const int col = (c & ~31) - (int)me * W, v0 = (c & 16) >> 2;   // chunk start, first 16-byte unit
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.f;
                for (int z = 0; z < nsplit; ++z) {
                    if (z == (int)me) {
                        uint32_t r[16];
                        tmem_ld16(tbase + c, r);
#pragma unroll
                        for (int e = 0; e < 16; ++e) acc[e] += __uint_as_float(r[e]);
                    } else {
                        const int slot = z - (z > (int)me ? 1 : 0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const uint4 u = lds128(unit_addr(slot, row, col, v0 + v));
                            acc[4 * v] += __uint_as_float(u.x);
                            acc[4 * v + 1] += __uint_as_float(u.y);
                            acc[4 * v + 2] += __uint_as_float(u.z);
                            acc[4 * v + 3] += __uint_as_float(u.w);
                        }
                    }
                }
                store_row16(acc, m, n0 + c);
            }
        }
    }

    // every role ends here.  After an abort, whichever role gave up: the
    // producer waits (bounded) for every copy it issued, so that none lands in
    // this CTA's shared memory after it exits, and the MMA issuer waits
    // (bounded) for the MMAs before TMEM is freed.
    if (warp == 0 && lane == 0 && *abort_flag) drain_copies();
    if (warp == 1 && lane == 0 && *abort_flag) {
        const uint64_t drain = global_timer() + timeout_ns;
        while (!mbar_try_wait(acc_done, 0) && global_timer() < drain) {
        }
    }
    tc_fence_before();
    if (PAIR)
        cluster_sync();   // neither CTA leaves while the other may still signal it or read its stages
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                         : "memory");
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

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *gaddr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(gaddr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_attr_done[7][kMaxDevices];
std::atomic<int> g_attr_done_grouped[2][kMaxDevices];
std::atomic<int> g_attr_done_pair[4][kMaxDevices];   // CTA-pair instances: (8-bit) * 2 + (TM == 256)
std::atomic<int> g_sms[kMaxDevices];
// clusters of 2, 4, 8 CTAs that can be resident at once, per code width (0: not yet asked; -1: none)
std::atomic<int> g_max_clusters[3][3][kMaxDevices];

}  // namespace

bool qmm_supported(const MatmulArgs &a) {
    return (a.bits == 4 || a.bits == 8) && a.K % 512 == 0 && a.M >= 1 && a.N >= 1 && encode_fn() != nullptr &&
           (reinterpret_cast<uintptr_t>(a.scales) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.biases) & 15) == 0;
}

namespace {
// Rows of W per CTA when K is not split: 224 where that takes no more waves of
// CTAs than 256 and so lowers the busiest SM's work (M = 2048 over 4096 rows of W:
// 128 tiles of 256 leave 24 of 152 SMs idle, 152 tiles of 224 fill them).
int qmm_tile_n(int64_t n_rows, int64_t row_tiles, int sms) {
    if (sms <= 0) return kTileN;
    auto cost = [&](int tn) {
        const int64_t tiles = (n_rows + tn - 1) / tn * row_tiles;
        return (tiles + sms - 1) / sms * tn;
    };
    return cost(224) < cost(kTileN) ? 224 : kTileN;
}

// CTA pairs (each W tile converted once per 2 TM rows of x) without a K split and
// without x converted once, where the row tiles pair up with at most one padding
// tile in five
bool qmm_pair(int64_t M, int tm, int split) {
    const int64_t mtiles = (M + tm - 1) / tm;
    return split == 1 && mtiles >= 2 && (mtiles % 2 == 0 || mtiles >= 5);
}

// g_attr_done slot of a kernel instance without the expert index
template <int BITS, bool XPRE, int TM>
constexpr int attr_slot() {
    return (BITS == 8 && TM == 256) ? 4 : (BITS == 4 && TM == 128) ? 5 + (int)XPRE : (BITS == 8 ? 1 : 0) + (XPRE ? 2 : 0);
}
// K split across a cluster of 2, 4 or 8 CTAs when the output has too few tiles to
// occupy half the SMs (prefill at M = 256), as many as still fit in one wave.
// Decided on the tiles of the kernel without the workspace, so that both
// variants split alike (same summation order, same bits).  Also records the
// device's SM count.
template <int BITS, int TM = (BITS == 4 ? 256 : 128)>
int qmm_split(const MatmulArgs &a, int dev) {
    using C = Cfg<BITS, false, TM>;
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K;
    int sms = g_sms[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();   // no split; the launch reports the device's state
            return 1;
        }
        g_sms[dev].store(sms, std::memory_order_relaxed);
    }
    const int64_t tiles = (int64_t)((N + kTileN - 1) / kTileN) * ((M + C::kTileM - 1) / C::kTileM);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = a.stream;
    int split = 1;
    if (2 * tiles <= sms) {
        for (int si = 2; si >= 0 && split == 1; --si) {
            const int S = 2 << si;
            if (S > K / (kGroup * kSBGroups) || tiles * S > sms) continue;
            const int bb = BITS == 8 ? 1 : (TM == 128 ? 2 : 0);
            constexpr int ab = attr_slot<BITS, false, TM>();
            int n = g_max_clusters[bb][si][dev].load(std::memory_order_relaxed);
            if (n == 0) {
                using C0 = C;
                if (!g_attr_done[ab][dev].load(std::memory_order_acquire)) {
                    if (cudaFuncSetAttribute(qmm_kernel<BITS, false, false, TM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C0::kSmemBytes) != cudaSuccess)
                        cudaGetLastError();
                    else
                        g_attr_done[ab][dev].store(1, std::memory_order_release);
                }
                cudaLaunchConfig_t q = cfg;
                q.dynamicSmemBytes = C0::kSmemBytes;
                q.gridDim = dim3(1, 1, (unsigned)S);
                cudaLaunchAttribute ca;
                ca.id = cudaLaunchAttributeClusterDimension;
                ca.val.clusterDim.x = 1;
                ca.val.clusterDim.y = 1;
                ca.val.clusterDim.z = (unsigned)S;
                q.attrs = &ca;
                q.numAttrs = 1;
                if (cudaOccupancyMaxActiveClusters(&n, qmm_kernel<BITS, false, false, TM>, &q) != cudaSuccess || n < 1) {
                    cudaGetLastError();   // the query's error is not the caller's
                    n = -1;
                }
                g_max_clusters[bb][si][dev].store(n, std::memory_order_relaxed);
            }
            if (n >= tiles) split = S;
        }
    }
    return split;
}

// split: K split across a cluster of this many CTAs (qmm_split)
// tn: rows of W per CTA (kTileN, or 224 without a K split; see qmm_tile_n)
// PAIR: CTA pairs along M sharing each W tile (no K split; see qmm_kernel)
template <int BITS, bool XPRE, int TM = (BITS == 4 ? 256 : 128), bool PAIR = false, int TN = kTileN>
cudaError_t launch_qmm_bits(const MatmulArgs &a, int dev, int split, int tn = kTileN) {
    using C = Cfg<BITS, XPRE, TM, PAIR, TN>;
    static std::atomic<int> attr_done_tn[kMaxDevices];   // the instance laid out for 224 rows
    std::atomic<int> &attr_done =
        TN != kTileN ? attr_done_tn[dev]
        : PAIR       ? g_attr_done_pair[(BITS == 8 ? 2 : 0) + (TM == 256 ? 1 : 0)][dev]
                     : g_attr_done[attr_slot<BITS, XPRE, TM>()][dev];
    if (TN != kTileN && tn != TN) return cudaErrorInvalidConfiguration;
    if (!attr_done.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(qmm_kernel<BITS, false, XPRE, TM, PAIR, TN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.store(1, std::memory_order_release);
    }
    if (PAIR && split != 1) return cudaErrorInvalidConfiguration;
    const uint32_t wbox = (uint32_t)(PAIR ? tn / 2 : tn);   // rows of W one CTA loads
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K, G = K / 64;
    if (XPRE) {
        const int64_t vecs = (int64_t)M * K / 8;
        cudaError_t e = launch_plain(x_to_f16_kernel<BITS>, dim3((unsigned)std::min<int64_t>((vecs + 255) / 256, 4096)),
                                     dim3(256), a.stream, static_cast<const uint4 *>(a.x), static_cast<uint4 *>(a.xf16),
                                     vecs);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tx, tw, ts, tb;
    if (!encode_2d(&tx, XPRE ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, XPRE ? a.xf16 : a.x, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, kGroup,
                   C::kTileM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.w, (uint64_t)K * BITS / 32, (uint64_t)N,
                   (uint64_t)K * BITS / 8, C::kRowWords, wbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, (uint64_t)G, (uint64_t)N, (uint64_t)G * 2, kSBGroups,
                   wbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.biases, (uint64_t)G, (uint64_t)N, (uint64_t)G * 2, kSBGroups,
                   wbox, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (split > 1 && tn != kTileN) return cudaErrorInvalidConfiguration;   // the K split owns 256 / split columns
    cudaLaunchConfig_t cfg = {};
    const int64_t mtiles = (M + C::kTileM - 1) / C::kTileM, ntiles = (N + tn - 1) / tn;
    // row tiles of x fastest where W has more bytes than x (see qmm_kernel)
    const int mfast = (int64_t)N * BITS / 8 > (int64_t)M * 2 && ntiles <= 65535 ? 1 : 0;
    const int64_t gx = mfast ? (PAIR ? (mtiles + 1) / 2 * 2 : mtiles) : (PAIR ? 2 * ntiles : ntiles);
    const int64_t gy = mfast ? ntiles : (PAIR ? (mtiles + 1) / 2 : mtiles);
    if (gy > 65535) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3((unsigned)gx, (unsigned)gy, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.pdl || XPRE) {   // with XPRE the launch before is the conversion of x into the workspace
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (split > 1) {
        cfg.gridDim.z = (unsigned)split;
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = (unsigned)split;
        ++na;
    } else if (PAIR) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)na;
    return cudaLaunchKernelEx(&cfg, qmm_kernel<BITS, false, XPRE, TM, PAIR, TN>, tx, tw, ts, tb, static_cast<__nv_bfloat16 *>(a.y), M,
                              N, K, (unsigned long long)a.timeout_ns, a.status, (const int *)nullptr,
                              a.debug_skip_copy ? 1 : 0, tn, mfast, 0);
}
}  // namespace

cudaError_t launch_qmm(const MatmulArgs &a) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (a.bits == 4) {
        const int split = qmm_split<4>(a, dev);
        const int sms = g_sms[dev].load(std::memory_order_relaxed);
        // few 256-row tiles (prefill at M = 256 over 4096 x 14336): 128-row tiles, where
        // they keep the K split (so that no CTA converts more of W) and still fit one
        // wave, put more SMs to work; the same choice with and without the workspace
        // (same summation order, same bits)
        const int64_t ntiles = (a.N + kTileN - 1) / kTileN;
        const int64_t tiles256 = ntiles * ((a.M + 255) / 256), tiles128 = ntiles * ((a.M + 127) / 128);
        if (sms > 0 && 4 * tiles256 * split <= 3 * (int64_t)sms && tiles128 * split <= sms &&
            qmm_split<4, 128>(a, dev) == split)
            return a.xf16 ? launch_qmm_bits<4, true, 128>(a, dev, split) : launch_qmm_bits<4, false, 128>(a, dev, split);
        const int tn = split == 1 ? qmm_tile_n(a.N, (a.M + 255) / 256, sms) : kTileN;
        if (!a.xf16 && qmm_pair(a.M, 256, split)) return launch_qmm_bits<4, false, 256, true>(a, dev, split, tn);
        return a.xf16 ? launch_qmm_bits<4, true>(a, dev, split, tn) : launch_qmm_bits<4, false>(a, dev, split, tn);
    }
    const int split = qmm_split<8>(a, dev);
    const int sms = g_sms[dev].load(std::memory_order_relaxed);
    const int tn128 = split == 1 ? qmm_tile_n(a.N, (a.M + 127) / 128, sms) : kTileN;
    const bool pair128 = qmm_pair(a.M, 128, split);
    if (!a.xf16) {
        if (qmm_pair(a.M, 256, split))
            return launch_qmm_bits<8, false, 256, true>(a, dev, split, qmm_tile_n(a.N, (a.M + 255) / 256, sms));
        return pair128 ? launch_qmm_bits<8, false, 128, true>(a, dev, split, tn128)
                       : launch_qmm_bits<8, false>(a, dev, split, tn128);
    }
    // x converted once: 256-row tiles where that needs no split and still fills half the
    // SMs (M = 2048 on 14336 x 4096: 743 -> 1205 TFLOP/s; on 4096 x 14336 one wave of
    // 128 such tiles against 1.7 waves of 128-row tiles)
    const int64_t tiles256 = ((a.N + kTileN - 1) / kTileN) * ((a.M + 255) / 256);
    if (split == 1 && sms > 0 && 2 * tiles256 >= sms) {
        // where 224-row W tiles fill the waves better, stages laid out for 224 rows:
        // three converted stages fit instead of two (M = 2048 on 4096 x 14336: 191.2 ->
        // 188.3 us; forcing 224-row tiles on 14336 x 4096 adds a wave, 187 -> 225 us)
        const int tn = qmm_tile_n(a.N, (a.M + 255) / 256, sms);
        if (tn == 224) return launch_qmm_bits<8, true, 256, false, 224>(a, dev, split, 224);
        return launch_qmm_bits<8, true, 256>(a, dev, split, tn);
    }
    return launch_qmm_bits<8, true>(a, dev, split, tn128);
}

// ---------------------------------------------------------------- expert-indexed matmul

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanMinTileM = 128;   // the smaller x tile of the two code widths (bounds the plan)

// One CTA: checks the indices (token in [0, T), expert in [0, E), experts
// non-decreasing), counts the rows of every expert and writes the work tiles
// {expert, first row, rows, 0} of at most tile_m rows each, in expert order,
// after the tile count.  Bad indices: a count of 0 (the matmul then does
// nothing) and AQ_DEVICE_STATUS_BAD_INDEX in the status word.
__global__ void __launch_bounds__(kPlanThreads, 1)
gather_plan_kernel(const int *__restrict__ lhs, const int *__restrict__ rhs, int R, int T, int E, int tile_m,
                   int *__restrict__ plan, int *status) {
    __shared__ int cnt[kMaxExperts];
    __shared__ int bad;
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    if (tid == 0) bad = 0;
    __syncthreads();
    for (int r = tid; r < R; r += blockDim.x) {
        const int l = __ldg(lhs + r), e = __ldg(rhs + r);
        if (l < 0 || l >= T || e < 0 || e >= E || (r > 0 && __ldg(rhs + r - 1) > e))
            bad = 1;
        else
            atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            plan[0] = 0;
            atomicExch(status, AQ_DEVICE_STATUS_BAD_INDEX);
        }
        return;
    }
    __shared__ int tile_off[kMaxExperts], row_off[kMaxExperts];
    if (tid == 0) {
        int tiles = 0, rows = 0;
        for (int e = 0; e < E; ++e) {
            tile_off[e] = tiles;
            row_off[e] = rows;
            tiles += (cnt[e] + tile_m - 1) / tile_m;
            rows += cnt[e];
        }
        plan[0] = tiles;
    }
    __syncthreads();
    int4 *tiles = reinterpret_cast<int4 *>(plan + kPlanHeaderInts);
    for (int e = tid; e < E; e += blockDim.x)
        for (int i = 0; i * tile_m < cnt[e]; ++i)
            tiles[tile_off[e] + i] = make_int4(e, row_off[e] + i * tile_m, min(tile_m, cnt[e] - i * tile_m), 0);
}

// x rows in row order of the matmul, converted once to the tensor-core
// kernel's fp16 chunk order: xg[r] = f16(x[lhs[r]]) (zeros for an index out
// of range, which the plan kernel reports), 16 bytes per thread and step.
template <int BITS>
__global__ void gather_rows_kernel(const uint4 *__restrict__ x, const int *__restrict__ lhs, uint4 *__restrict__ xg,
                                   int R, int T, int row_vecs) {
    griddep_launch();   // the expert-indexed matmul after it may start its set-up (it waits for xg)
    const int64_t total = (int64_t)R * row_vecs;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / row_vecs, c = i - r * row_vecs;
        const int l = __ldg(lhs + r);
        xg[i] = (l >= 0 && l < T) ? x_chunk_f16<BITS>(__ldg(x + (int64_t)l * row_vecs + c)) : make_uint4(0u, 0u, 0u, 0u);
    }
}

int64_t plan_max_tiles(int64_t R, int64_t E) { return (R + kPlanMinTileM - 1) / kPlanMinTileM + E; }
int64_t plan_bytes(int64_t R, int64_t E) { return (kPlanHeaderInts * 4 + 16 * plan_max_tiles(R, E) + 127) & ~int64_t(127); }

template <int BITS>
cudaError_t launch_gather_bits(const GatherArgs &g, int dev, int sms) {
    using C = Cfg<BITS, true>;
    // rows of W per CTA on the row-tile count without the experts' partial tiles
    const int tn = qmm_tile_n(g.N, (g.R + C::kTileM - 1) / C::kTileM, sms);
    // Two launches: the row tiles that fill whole waves of CTAs, one CTA per output
    // tile, then the rest with K split across the two CTAs of a cluster (256-row W
    // tiles), so the last, partly filled wave takes half as long.  Counted on the
    // expected row-tile count (each expert adds about half a partial tile); the
    // plan's actual tiles decide which CTAs run (past the count, a CTA exits at once).
    // The Mixtral-shaped down projection (4096 x 14336 experts): 16 row tiles x 19 W
    // tiles of 224 rows in two full waves, then 4 x 16 x 2 half-K CTAs.
    const int64_t max_tiles = (g.R + C::kTileM - 1) / C::kTileM + g.E;
    int64_t full = 0;   // row tiles of the first launch
    {
        const int64_t est = std::min<int64_t>((g.R + C::kTileM - 1) / C::kTileM + g.E / 2, max_tiles);
        const int64_t wt = (g.N + tn - 1) / tn;
        full = sms > 0 ? (est * wt / sms) * sms / wt : max_tiles;
        if (g.K % (2 * kGroup * kSBGroups) != 0) full = max_tiles;   // no even K split
        if (full > max_tiles) full = max_tiles;
    }
    const int bi = BITS == 8 ? 1 : 0;
    if (!g_attr_done_grouped[bi][dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(qmm_kernel<BITS, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        g_attr_done_grouped[bi][dev].store(1, std::memory_order_release);
    }
    const int R = (int)g.R, N = (int)g.N, K = (int)g.K, E = (int)g.E, G = K / 64;
    int *plan = static_cast<int *>(g.workspace);
    void *xg = static_cast<uint8_t *>(g.workspace) + plan_bytes(g.R, g.E);
    cudaError_t e = launch_plain(gather_plan_kernel, dim3(1), dim3(kPlanThreads), g.stream, g.lhs, g.rhs, R,
                                 (int)g.T, E, (int)C::kTileM, plan, g.status);
    if (e != cudaSuccess) return e;
    e = launch_plain(gather_rows_kernel<BITS>, dim3((unsigned)(sms * 4)), dim3(256), g.stream,
                     static_cast<const uint4 *>(g.x), g.lhs, static_cast<uint4 *>(xg), R, (int)g.T, K / 8);
    if (e != cudaSuccess) return e;
    CUtensorMap tx, tw, ts, tb;
    if (!encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xg, (uint64_t)K, (uint64_t)R, (uint64_t)K * 2, kGroup,
                   C::kTileM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, g.w, (uint64_t)K * BITS / 32, (uint64_t)E * N,
                   (uint64_t)K * BITS / 8, C::kRowWords, (uint32_t)tn, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, g.scales, (uint64_t)G, (uint64_t)E * N, (uint64_t)G * 2,
                   kSBGroups, (uint32_t)tn, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, g.biases, (uint64_t)G, (uint64_t)E * N, (uint64_t)G * 2,
                   kSBGroups, (uint32_t)tn, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // programmatic launches: after the row gather, the plan (two launches back) is
    // complete and the kernel waits for the gathered rows before it reads them; the
    // second launch waits for the first in the same way.  With the K split, the two
    // CTAs of an output tile form a cluster.
    auto launch_part = [&](int64_t tile0, int64_t rows_tiles, int split, int tn_part,
                           const CUtensorMap &twp, const CUtensorMap &tsp, const CUtensorMap &tbp) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((N + tn_part - 1) / tn_part), (unsigned)rows_tiles, (unsigned)split);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = g.stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = (unsigned)split;
        cfg.attrs = attr;
        cfg.numAttrs = split > 1 ? 2 : 1;
        return cudaLaunchKernelEx(&cfg, qmm_kernel<BITS, true, true>, tx, twp, tsp, tbp,
                                  static_cast<__nv_bfloat16 *>(g.y), R, N, K, (unsigned long long)g.timeout_ns,
                                  g.status, (const int *)plan, 0, tn_part, 0, (int)tile0);
    };
    if (full > 0) {
        e = launch_part(0, full, 1, tn, tw, ts, tb);
        if (e != cudaSuccess || full == max_tiles) return e;
    }
    CUtensorMap tw2 = tw, ts2 = ts, tb2 = tb;   // W boxes of 256 rows for the split launch
    if (tn != kTileN &&
        (!encode_2d(&tw2, CU_TENSOR_MAP_DATA_TYPE_UINT32, g.w, (uint64_t)K * BITS / 32, (uint64_t)E * N,
                    (uint64_t)K * BITS / 8, C::kRowWords, (uint32_t)kTileN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
         !encode_2d(&ts2, CU_TENSOR_MAP_DATA_TYPE_UINT16, g.scales, (uint64_t)G, (uint64_t)E * N, (uint64_t)G * 2,
                    kSBGroups, (uint32_t)kTileN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
         !encode_2d(&tb2, CU_TENSOR_MAP_DATA_TYPE_UINT16, g.biases, (uint64_t)G, (uint64_t)E * N, (uint64_t)G * 2,
                    kSBGroups, (uint32_t)kTileN, CU_TENSOR_MAP_SWIZZLE_NONE)))
        return cudaErrorInvalidValue;
    return launch_part(full, max_tiles - full, 2, kTileN, tw2, ts2, tb2);
}

}  // namespace

size_t gather_workspace_bytes(int64_t R, int64_t K, int64_t E) {
    return (size_t)(plan_bytes(R, E) + R * K * 2);
}

cudaError_t launch_gather_qmm(const GatherArgs &g) {
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
    if (!encode_fn()) return cudaErrorNotSupported;
    return g.bits == 8 ? launch_gather_bits<8>(g, dev, sms) : launch_gather_bits<4>(g, dev, sms);
}

}  // namespace aq
