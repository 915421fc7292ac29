// The consumer side of the weight-streaming kernels (qmv_tma.cu and
// qmv_chain.cu): one warp's share of a shared-memory stage, i.e. 16 rows of W
// times one 256-code column block (4 groups of 64), folded into the warp's
// fp32 accumulators.  Internal header (not installed).
//
// Arithmetic per group g and row n (fp32 accumulation):
//   D[n,m,g] = sum_{k in g} (128 + q[n,k]) * x[m,k]      (mma.sync, exact bf16 operands)
//   acc     += scale[n,g] * D + (bias[n,g] - 128*scale[n,g]) * X[m,g],   X = sum_{k in g} x
// MMA A rows are W rows (r0 = lane/4 and r1 = r0 + 8); B columns are rows of x
// (column lane/4 for B, columns 2*(lane%4) and +1 for the accumulators).
#pragma once

#include "aq_ptx.cuh"

namespace aq {
namespace qmv {
namespace {

using namespace dev;

constexpr int kRows = 16;                                  // rows of W per tile (MMA M)
constexpr int kConsumerWarps = 8;
constexpr int kBlockCodes = 256;                           // codes per column block (one 128-byte swizzle row)
constexpr int kStageCodes = kBlockCodes * kConsumerWarps;  // 2048 codes per stage
constexpr int kStageGroups = kStageCodes / 64;             // 32
constexpr int kCodeBlockBytes = kRows * 128;               // 2048
constexpr int kCodesBytes = kCodeBlockBytes * kConsumerWarps;  // 16384
constexpr int kSBBytes = kRows * kStageGroups * 2;         // 1024 (scales, and again biases)
constexpr int kStageBytes = kCodesBytes + 2 * kSBBytes;    // 18432

// Per-thread shared-memory addresses, fixed while one matrix is processed.
struct ConsumerThread {
    uint32_t caddr[4];  // codes of row r0, group g, word pair 2j..2j+1, relative to the block base (swizzle undone)
    uint32_t x_row;     // permuted x, row min(lane/4, M-1), this warp's block and word pair (absolute)
    uint32_t xsum;      // per-group sums of x for column 2j (absolute); column 2j+1 at +G*4
    int G;
    bool xs0_ok, xs1_ok;
};

__device__ __forceinline__ void consumer_init(ConsumerThread &c, int warp, int lane, uint32_t x_s, uint32_t xsum_s,
                                              int M, int K) {
    const int gid = lane >> 2, j = lane & 3;
#pragma unroll
    for (int g = 0; g < 4; ++g)
        c.caddr[g] = (uint32_t)(gid * 128 + ((((2 * g + (j >> 1)) ^ gid) << 4) | ((j & 1) << 3)));
    // B columns beyond M read a real row: those accumulator columns are never used
    const int xr = gid < M ? gid : M - 1;
    c.x_row = x_s + (uint32_t)(xr * K * 2 + warp * 512 + 2 * j * 16);
    c.G = K >> 6;
    c.xsum = xsum_s + (uint32_t)((2 * j < M ? 2 * j : 0) * c.G * 4 + warp * 16);
    c.xs0_ok = 2 * j < M;
    c.xs1_ok = 2 * j + 1 < M;
}

// Adds one 16-row x 256-code column block (column block kb*8 + warp of the
// matrix) to acc.  `codes` is the block's 128-byte-swizzled code tile (16
// rows of 128 bytes); `sc` points at the scales of row lane/4 for the block's
// 4 groups, row lane/4 + 8 at +S_R1 bytes, and the biases at +B_OFF.
template <bool ONE_ROW, int S_R1, int B_OFF>
__device__ __forceinline__ void consume_block(uint32_t codes, uint32_t sc, int kb, const ConsumerThread &c,
                                              float (&acc)[4]) {
    const uint32_t magic = kMagic;
    const uint2 s0 = lds64(sc), s1 = lds64(sc + S_R1);
    const uint2 b0 = lds64(sc + B_OFF), b1 = lds64(sc + B_OFF + S_R1);
    const uint32_t xb = c.x_row + (uint32_t)kb * (kConsumerWarps * 512);
    const uint32_t xsb = c.xsum + (uint32_t)kb * (kConsumerWarps * 16);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint2 w0 = lds64(codes + c.caddr[g]);
        const uint2 w1 = lds64(codes + c.caddr[g] + 1024);
        float d[4];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t wa = i ? w0.y : w0.x;
            const uint32_t wb = i ? w1.y : w1.x;
            const uint4 X = lds128(xb + g * 128 + i * 16);
            const uint32_t wa4 = wa >> 4, wb4 = wb >> 4, wa8 = wa >> 8, wb8 = wb >> 8;
            const uint32_t wa12 = wa >> 12, wb12 = wb >> 12;
            if (i == 0)
                mma_bf16_16816_zc(d, code_pair(wa, magic), code_pair(wb, magic), code_pair(wa4, magic),
                                  code_pair(wb4, magic), X.x, X.y);
            else
                mma_bf16_16816(d, code_pair(wa, magic), code_pair(wb, magic), code_pair(wa4, magic),
                               code_pair(wb4, magic), X.x, X.y);
            mma_bf16_16816(d, code_pair(wa8, magic), code_pair(wb8, magic), code_pair(wa12, magic),
                           code_pair(wb12, magic), X.z, X.w);
        }
        const uint32_t sw0 = (g < 2) ? s0.x : s0.y, sw1 = (g < 2) ? s1.x : s1.y;
        const uint32_t bw0 = (g < 2) ? b0.x : b0.y, bw1 = (g < 2) ? b1.x : b1.y;
        const float2 sc2 = make_float2((g & 1) ? bf16hi(sw0) : bf16lo(sw0), (g & 1) ? bf16hi(sw1) : bf16lo(sw1));
        const float2 p = fma2(make_float2(-128.f, -128.f), sc2,
                              make_float2((g & 1) ? bf16hi(bw0) : bf16lo(bw0), (g & 1) ? bf16hi(bw1) : bf16lo(bw1)));
        if (ONE_ROW) {
            const float xs = lds_f32(xsb + g * 4);
            const float2 a02 = fma2(sc2, make_float2(d[0], d[2]), fma2(p, make_float2(xs, xs), make_float2(acc[0], acc[2])));
            acc[0] = a02.x;
            acc[2] = a02.y;
        } else {
            const float xs0 = c.xs0_ok ? lds_f32(xsb + g * 4) : 0.f;
            const float xs1 = c.xs1_ok ? lds_f32(xsb + c.G * 4 + g * 4) : 0.f;
            const float2 xs = make_float2(xs0, xs1);
            const float2 a01 = fma2(make_float2(sc2.x, sc2.x), make_float2(d[0], d[1]),
                                    fma2(make_float2(p.x, p.x), xs, make_float2(acc[0], acc[1])));
            const float2 a23 = fma2(make_float2(sc2.y, sc2.y), make_float2(d[2], d[3]),
                                    fma2(make_float2(p.y, p.y), xs, make_float2(acc[2], acc[3])));
            acc[0] = a01.x;
            acc[1] = a01.y;
            acc[2] = a23.x;
            acc[3] = a23.y;
        }
    }
}

// Layout of a shared stage (16 rows x 2048 codes + scales/biases of 32 groups):
// warp w's block codes at +w*2048, scales row r at +16384 + r*64 + 8*w.
template <bool ONE_ROW>
__device__ __forceinline__ void consume_shared_stage(uint32_t st, int warp, int lane, int kb, const ConsumerThread &c,
                                                     float (&acc)[4]) {
    consume_block<ONE_ROW, 512, kSBBytes>(st + (uint32_t)(warp * kCodeBlockBytes),
                                          st + (uint32_t)(kCodesBytes + (lane >> 2) * 64 + 8 * warp), kb, c, acc);
}

}  // namespace
}  // namespace qmv
}  // namespace aq
