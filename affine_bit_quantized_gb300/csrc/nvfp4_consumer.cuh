// The consumer side of the NVFP4 weight-streaming kernels (nvfp4_qmv.cu and
// the NVFP4 mode of qmv_chain.cu).  Internal header (not installed).
//
// Format (the NVFP4 layout of NVIDIA's model optimizer, the mode=nvfp4,
// group_size=16 checkpoint of the "MLX CUDA Cleanup Plan" page, Refactor Plan
// Phase 3b): FP4 E2M1 codes packed eight per uint32 (lowest nibble = lowest
// k), one FP8 E4M3 scale per 16 codes along K, one fp32 scale per tensor:
//
//     w[n,k] = global * e4m3(scale[n, k/16]) * e2m1(q[n,k])
//
// A stage holds 32 rows of W x 2048 codes (eight 128-byte-swizzled code boxes,
// as in the 4-bit affine kernels) and the 32 x 128 E4M3 scale bytes of those
// codes (one 128-byte-swizzled box); consumer warp w takes the 128-code column
// block w of every stage.  Arithmetic:
//
//  * e2m1 * e4m3 has at most six significant bits and lies in [2^-10, 2688],
//    so a code pair converted to fp16 (cvt.rn.f16x2.e2m1x2) times its block
//    scale (fp16, exact for every finite E4M3 value) is the exact weight in
//    fp16: no per-group fold, the MMA accumulates across all groups;
//  * x is staged in fp16, each row scaled by a power of two so that its bf16
//    values stay exact; the partial sums are scaled back and the reducer
//    multiplies by the tensor scale before the one bf16 rounding;
//  * lane (g, t) of a warp holds 32 consecutive codes of each of its four W
//    rows g + 8r (one 16-byte load per row), i.e. two whole scale groups; MMA
//    step s takes bytes 2s and 2s+1 of those 16, and the x fragment of step s
//    is the four x values at the same code positions, so A and B agree on
//    which k sits in each MMA slot.
//
// Staged x order within a 128-code block (256 bytes of fp16): code c goes to
// byte ((c % 32) / 4) * 32 + (c / 32) * 8 + (c % 4) * 2, so that at step s the
// four lanes t of one x row read 32 consecutive bytes.  With rows 16 bytes
// apart modulo 128 (a pad per row), the eight rows of a warp's 8-byte loads
// then cover every bank exactly twice: two shared-memory wavefronts per load,
// the least 256 bytes can take.  (In natural order lanes t and t + 2 of a row
// hit the same banks, which doubles that.)
#pragma once

#include <cuda_bf16.h>

#include "aq_ptx.cuh"
#include "qmv_consumer.cuh"

namespace aq {
namespace qmv {
namespace {

using namespace dev;

constexpr int kNvCodes = 2048;                          // codes per row and stage (1024 bytes)
constexpr int kNvScaleBytes = kRows * (kNvCodes / 16);  // 4096: one E4M3 byte per 16 codes, 32 rows
constexpr int kNvStage = kCodesBytes + kNvScaleBytes;   // 36864
static_assert(kNvStage == kStageBytes, "an NVFP4 stage fills an affine stage's room exactly");

// fp16x2 of the two E2M1 codes of byte `B` of v (low nibble in the low half)
template <int B>
__device__ __forceinline__ uint32_t e2m1_pair(uint32_t v) {
    uint32_t r;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b%2;\n}"
        : "=r"(r)
        : "r"(v), "n"(B));
    return r;
}
// fp16x2 of the two E4M3 bytes in the low 16 bits of v (low byte in the low half)
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t v) {
    uint32_t r;
    asm("{\n .reg .b16 h;\n cvt.u16.u32 h, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}" : "=r"(r) : "r"(v));
    return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
__device__ __forceinline__ uint32_t lds16u(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts64u(uint32_t a, uint32_t x, uint32_t y) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}

// Byte offset, within its 256-byte block, of the 16-byte word iw (codes
// 8 iw .. 8 iw + 7) of a 128-code block in the staged order: its first four
// codes; the other four sit 32 bytes further on.
__device__ __forceinline__ uint32_t nv_x_word_offset(int iw) { return (uint32_t)((iw & 3) * 64 + (iw >> 2) * 8); }

// Per-thread shared-memory offsets of the NVFP4 consumer.
struct NvThread {
    uint32_t code[4];   // stage offsets of the lane's 16 code bytes in W rows g + 8r
    uint32_t sb;        // offset of its two scale bytes in row g of the scale box (rows + 8r at + 1024 r)
};

__device__ __forceinline__ void nv_consumer_init(NvThread &c, int warp, int lane) {
    const int gid = lane >> 2, t = lane & 3;
    // 128-byte swizzle: 16-byte unit u of box row r sits at unit u ^ (r % 8)
#pragma unroll
    for (int r = 0; r < 4; ++r)
        c.code[r] = (uint32_t)((warp >> 1) * kBoxBytes + (gid + 8 * r) * 128 + (((4 * (warp & 1) + t) ^ gid) << 4));
    // scale bytes of groups warp*8 + 2t, +1 of row gid (unit warp/2 of the 128-byte row)
    c.sb = (uint32_t)(gid * 128 + (((warp >> 1) ^ gid) << 4) + 8 * (warp & 1) + 2 * t);
}

// Adds warp `warp`'s block of a stage (32 W rows x 128 codes) to acc.  xq: the
// byte address of the lane's first x fragment in the staged block, i.e. block
// base + row offset + t * 8 (staged order above).
__device__ __forceinline__ void consume_stage_nvfp4(uint32_t st, const NvThread &c, uint32_t xq,
                                                    float (&acc)[2][4]) {
    uint4 cw[4];
    uint32_t sa2[4], sb2[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        cw[r] = lds128(st + c.code[r]);
        // the block scales of the lane's two groups in row gid + 8r, each in both halves
        const uint32_t s2 = e4m3_pair(lds16u(st + kCodesBytes + c.sb + 8 * 128 * r));
        sa2[r] = prmt(s2, s2, 0x1010u);
        sb2[r] = prmt(s2, s2, 0x3232u);
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const uint2 X = lds64(xq + s * 32);   // x at the lane's codes 4s .. 4s+3
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 &R0 = cw[2 * h], &R1 = cw[2 * h + 1];   // rows gid + 16h, gid + 8 + 16h
            const uint32_t w0 = s < 2 ? R0.x : s < 4 ? R0.y : s < 6 ? R0.z : R0.w;
            const uint32_t w1 = s < 2 ? R1.x : s < 4 ? R1.y : s < 6 ? R1.z : R1.w;
            const uint32_t g0 = s < 4 ? sa2[2 * h] : sb2[2 * h];
            const uint32_t g1 = s < 4 ? sa2[2 * h + 1] : sb2[2 * h + 1];
            uint32_t a0, a1, a2, a3;
            if (s & 1) {
                a0 = hmul2(e2m1_pair<2>(w0), g0);
                a1 = hmul2(e2m1_pair<2>(w1), g1);
                a2 = hmul2(e2m1_pair<3>(w0), g0);
                a3 = hmul2(e2m1_pair<3>(w1), g1);
            } else {
                a0 = hmul2(e2m1_pair<0>(w0), g0);
                a1 = hmul2(e2m1_pair<0>(w1), g1);
                a2 = hmul2(e2m1_pair<1>(w0), g0);
                a3 = hmul2(e2m1_pair<1>(w1), g1);
            }
            mma_f16_16816(acc[h], a0, a1, a2, a3, X.x, X.y);
        }
    }
}

// Stages this warp's slice of x [M][K] (bf16 in global memory, read through
// L2) for the NVFP4 consumer: the 128-code blocks kb * 16 + warp of every row,
// fp16 in the staged order, block kb of row m at
//     xs.xq + warp * xs.wq + m * xw_row_bytes(M, KB, 4) + kb * 256,
// with the same per-warp power-of-two row scales as stage_x_warp (which this
// mirrors without the group sums: NVFP4 needs no fold).  Sets inv[c] = 2^-e
// of the x row of MMA column 2j + c (j = lane % 4).  M * KB * 4096 <= 32768.
template <bool ONE_ROW>
__device__ __forceinline__ void stage_x_nv_warp(const XStage &xs, const __nv_bfloat16 *xg, int M_, int K, int warp,
                                                int lane, float (&inv)[2]) {
    constexpr int MR = ONE_ROW ? 1 : kMaxM;
    const int M = ONE_ROW ? 1 : M_;
    const int nblk = K / 128;
    const int KB = (K + kNvCodes - 1) / kNvCodes;
    const int kbw = warp < nblk ? (nblk - warp + kConsumerWarps - 1) / kConsumerWarps : 0;
    const int wpr = kbw * 16;   // 16-byte words of a row in the slice
    const int words = M * wpr;
    const uint32_t xq = xs.xq + (uint32_t)(warp * xs.wq);
    const int xrb = xw_row_bytes(M, KB, 4);
    constexpr int NW = kMaxXBytes / 16 / kConsumerThreads;
    uint4 v[NW];
    int row[NW];
#pragma unroll
    for (int u = 0; u < NW; ++u) {
        const int wi = u * 32 + lane;
        row[u] = 0;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (wi < words) {
            const int m = ONE_ROW ? 0 : wi / wpr, r = wi - m * wpr;
            const int kb = r >> 4, iw = r & 15;
            row[u] = m;
            v[u] = ldg_cg_v4(xg + (size_t)m * K + (size_t)(kb * kConsumerWarps + warp) * 128 + iw * 8);
        }
    }
    int e[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
        int mx = 0;
#pragma unroll
        for (int u = 0; u < NW; ++u) {
            if (row[u] == m) {
                mx = max(mx, bf16x2_abs_max(v[u].x));
                mx = max(mx, bf16x2_abs_max(v[u].y));
                mx = max(mx, bf16x2_abs_max(v[u].z));
                mx = max(mx, bf16x2_abs_max(v[u].w));
            }
        }
        e[m] = x_scale_exponent(__reduce_max_sync(0xFFFFFFFFu, mx));
    }
    __syncwarp();   // every lane has finished reading the previous x from the region
#pragma unroll
    for (int u = 0; u < NW; ++u) {
        const int wi = u * 32 + lane;
        if (wi < words) {
            const int m = row[u];
            int em = e[0];
            if (!ONE_ROW) {
#pragma unroll
                for (int mm = 1; mm < MR; ++mm) em = m == mm ? e[mm] : em;
            }
            const int r = wi - m * wpr, kb = r >> 4, iw = r & 15;
            const float sc = pow2f(em);
            const uint4 a = v[u];
            const uint32_t q = xq + (uint32_t)(m * xrb + kb * 256) + nv_x_word_offset(iw);
            sts64u(q, f32x2_to_f16x2(bf16lo(a.x) * sc, bf16hi(a.x) * sc), f32x2_to_f16x2(bf16lo(a.y) * sc, bf16hi(a.y) * sc));
            sts64u(q + 32, f32x2_to_f16x2(bf16lo(a.z) * sc, bf16hi(a.z) * sc),
                   f32x2_to_f16x2(bf16lo(a.w) * sc, bf16hi(a.w) * sc));
        }
    }
    if (ONE_ROW) {
        inv[0] = inv[1] = pow2f(-e[0]);
    } else {
        const int j = lane & 3;
        const int r0 = 2 * j < M ? 2 * j : M - 1, r1 = 2 * j + 1 < M ? 2 * j + 1 : M - 1;
        int e0 = e[0], e1 = e[0];
#pragma unroll
        for (int mm = 1; mm < MR; ++mm) {
            e0 = r0 == mm ? e[mm] : e0;
            e1 = r1 == mm ? e[mm] : e1;
        }
        inv[0] = pow2f(-e0);
        inv[1] = pow2f(-e1);
    }
    __syncwarp();   // the region is written before any lane reads it
}

}  // namespace
}  // namespace qmv
}  // namespace aq
