// The consumer side of the weight-streaming kernels (qmv_tma.cu and
// qmv_chain.cu): staging of x in shared memory, one warp's share of a
// shared-memory stage (32 rows of W x one 128-code column block, i.e. two
// groups of 64; sixteen warps cover a 2048-code stage), and the per-tile
// cross-warp reduction.  Internal header (not installed).
//
// Arithmetic per group g, row n and row m of x (fp32 accumulation), for the
// warp w whose column blocks hold g:
//   x'[m,k]  = fp16(2^e[w,m] * x[m,k] / c[k]),  c[k] = 1 or 16 by position in its
//              8-element word (see below); e[w,m] puts the maximum of |x[m,k]|
//              over the warp's own slice of k in [2^14, 2^15)
//   D[n,m,g] = sum_{k in g} (1024 + c[k] * q[n,k]) * x'[m,k]     (mma.sync, exact fp16 operands)
//            = 1024 * X'[m,g] + 2^e[w,m] * sum_{k in g} q[n,k] * x[m,k]
//   acc_w   += scale[n,g] * (D - 1024 * X'[m,g]) + bias[n,g] * Xs[m,g]
//   y[m,n]   = sum over warps w, in warp order, of (2^-e[w,m] * acc_w)   (power-of-two scaling: exact)
// with X'[m,g] = sum_{k in g} x'[m,k] and Xs[m,g] = 2^e[w,m] * sum_{k in g} x[m,k].
//
// Codes become exact fp16 values with one LOP3 per pair: within a packed word
// the nibbles at bits 0-3 and 16-19 go into the mantissa as 1024 + q, those at
// bits 4-7 and 20-23 as 1024 + 16q (hence c = 16 there), and the word shifted
// right by 8 gives the other four codes the same way.  A bf16 value has an
// 8-bit significand, so with the power-of-two scale every element of x whose
// magnitude is within 2^-29 of the slice maximum is exact in fp16; smaller ones
// round to the fp16 subnormal grid, an absolute error below 2^-39 of the slice
// maximum.
//
// MMA A rows are W rows: row block h (0, 1) of the 32-row tile holds rows
// 16h + lane/4 and 16h + lane/4 + 8.  B columns are rows of x (column lane/4
// reads row min(lane/4, M-1); columns beyond M are never used).
#pragma once

#include <cuda_bf16.h>

#include "aq_ptx.cuh"

namespace aq {
namespace qmv {
namespace {

using namespace dev;

constexpr int kRows = 32;                                  // rows of W per tile
constexpr int kConsumerWarps = 16;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kBoxes = 8;                                  // code boxes per stage ({32 words, 32 rows})
constexpr int kBoxBytes = kRows * 128;                     // 4096
constexpr int kCodesBytes = kBoxes * kBoxBytes;            // 32768
constexpr int kSBRegion = 2048;                            // room for one scale (or bias) box per stage
constexpr int kStageBytes = kCodesBytes + 2 * kSBRegion;   // 36864

// Geometry by code width.  A stage is 32 rows x 1024 bytes of codes, i.e.
// 2048 4-bit or 1024 8-bit codes; each of the sixteen warps takes 128 bytes
// of every row (two groups of 4-bit codes, one group of 8-bit codes).
template <int BITS>
struct Geo {
    static_assert(BITS == 4 || BITS == 8, "4-bit and 8-bit codes");
    static constexpr int kGroupsPerWarp = BITS == 4 ? 2 : 1;
    static constexpr int kWarpCodes = 64 * kGroupsPerWarp;              // codes of a warp's column block
    static constexpr int kStageCodes = kWarpCodes * kConsumerWarps;     // 2048 or 1024
    static constexpr int kStageGroups = kStageCodes / 64;               // 32 or 16
    static constexpr int kBoxCodes = 1024 / BITS;                       // codes per 128-byte box row
    static constexpr int kSBRowBytes = kStageGroups * 2;                // 64 or 32 bytes: scale-box row
};
// the same numbers at run time (host and device)
__host__ __device__ constexpr int stage_codes(int bits) { return bits == 4 ? 2048 : 1024; }
__host__ __device__ constexpr int stage_groups(int bits) { return stage_codes(bits) / 64; }
constexpr int kMaxM = 8;                                   // rows of x per block of 8 MMA columns
constexpr int kMaxRows = 16;                               // rows of x with two blocks (single-matmul kernel)
constexpr int kMaxXBytes = 32768;                          // staging room for x (M * K * 2, K in whole stages)
constexpr int kXInfoBytes = 96;                            // int row_max[2][8], float inv_scale[8]
// Row stride of x staged in natural order (the NVFP4 kernel): 2K bytes, plus a
// 16-byte pad per row with several rows (rows 2K bytes apart would put the
// row addresses a warp reads at once in the same banks).
__host__ __device__ constexpr int x_row_bytes(int M, int K) { return M == 1 ? 2 * K : 2 * K + 16; }

// named barrier 1: the consumer warps only (the producer warp runs on)
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// Staged x of the current matmul, one region per consumer warp.  A warp reads
// only the x of its own column blocks (block kb * 16 + warp of every stage
// kb), so it stages that slice itself, with no barrier against the other
// warps: a warp may stage the next matmul's x while the others still work on
// the previous one, since the regions never overlap.  In the region of warp w
// (fragments at xq + w * wq, sums at xsum + w * ws):
//   fragments: row m at m * xw_row_bytes(M, KB); stage kb at kb * (groups per
//              warp) * 128; group gl at gl * 128; for word half i (words 2t+i
//              of the group, t = 0..3) a 64-byte "quad" at i * 64 holds four
//              16-byte rows (fragment register p = 0..3), each the registers
//              of threads t = 0..3, so one ldmatrix.x4 per quad serves all 32
//              lanes;
//   sums:      float2 (Xs, X') per row, stage and group, row m at
//              m * xsw_row_bytes(M, KB).
// KB is the matmul's (or K pass's) stage count; the regions are sized for the
// largest M * KB of the launch.
struct XStage {
    uint32_t xq, xsum;  // bases of the fragment and sum regions
    int wq, ws;         // bytes per warp of each
};
// Row strides inside a warp's region.  A fragment row is a multiple of 128
// bytes; with several rows, the eight row addresses of an ldmatrix (rows 0..7
// of x) would share banks, so one 16-byte pad per row shifts row m by m
// 16-byte bank groups.  One row needs no pad.  The sums are read once per
// group, so their rows go unpadded.
__host__ __device__ constexpr int xw_row_bytes(int M, int KB, int bits) {
    return KB * (bits == 4 ? 256 : 128) + (M == 1 ? 0 : 16);
}
__host__ __device__ constexpr int xsw_row_bytes(int M, int KB, int bits) { return KB * (bits == 4 ? 16 : 8); }
// Bytes per warp of the fragment and sum regions for x of up to x_bytes =
// M * KB * (stage codes) * 2 (the rounded-up size of x) and max_m rows.
__host__ __device__ constexpr int xw_region_bytes(int x_bytes, int max_m) {
    return x_bytes / kConsumerWarps + (max_m == 1 ? 0 : 16 * max_m);
}
__host__ __device__ constexpr int xsw_region_bytes(int x_bytes, int max_m) {
    return x_bytes / (16 * kConsumerWarps);
}
// M * K * 2 with K rounded up to whole stages: the staging room x needs
__host__ __device__ constexpr int x_stage_bytes(int M, int K, int bits) {
    return M * ((K + stage_codes(bits) - 1) / stage_codes(bits)) * stage_codes(bits) * 2;
}

__device__ __forceinline__ int x_scale_exponent(int max_bits) {
    // e with max|x| * 2^e in [2^14, 2^15); 0 for an all-zero row and for a row
    // holding inf or nan (propagated unchanged)
    if (max_bits == 0 || max_bits >= 0x7F80) return 0;
    const int e = 14 - ((max_bits >> 7) - 127);
    return e < -126 ? -126 : (e > 126 ? 126 : e);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }  // e in [-126, 127]

__device__ __forceinline__ int bf16x2_abs_max(uint32_t v) {
    const int a = (int)(v & 0x7FFFu), b = (int)((v >> 16) & 0x7FFFu);
    return a > b ? a : b;
}
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float f16x2_sum(uint32_t v) {
    float lo, hi;
    asm("{\n .reg .f16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}"
        : "=f"(lo), "=f"(hi)
        : "r"(v));
    return lo + hi;
}
__device__ __forceinline__ uint4 ldg_cg_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Stages this warp's slice of x [M][K] (bf16 in global memory, read through L2,
// rows ldx elements apart): fragments and (Xs, X') of the column blocks
// kb * 16 + warp, kb < KB, of every row.  The power-of-two scale 2^e of a row
// comes from the maximum over the warp's own slice; each warp unscales its
// own partial sums (write_partials), so warps need not agree on e.  Sets
// inv[c] = 2^-e of the x row of MMA column 2j + c (j = lane % 4; row 0 when
// ONE_ROW).  Only the calling warp takes part.  M * KB * (stage codes) * 2
// <= XROOM (the region's room), K % 64 == 0.
template <int BITS, bool ONE_ROW, int XROOM = kMaxXBytes, int NB = 1>
__device__ __forceinline__ void stage_x_warp(const XStage &xs, const __nv_bfloat16 *xg, int M_, int K, int ldx,
                                             int warp, int lane, float (&inv)[2 * NB]) {
    constexpr int MR = ONE_ROW ? 1 : 8 * NB;   // rows of x staged at most
    using Gm = Geo<BITS>;
    const int M = ONE_ROW ? 1 : M_;
    const int nblk = K / Gm::kWarpCodes;                          // column blocks of K
    const int KB = (K + Gm::kStageCodes - 1) / Gm::kStageCodes;   // stages
    const int kbw = warp < nblk ? (nblk - warp + kConsumerWarps - 1) / kConsumerWarps : 0;
    constexpr int WPS = Gm::kGroupsPerWarp * 8;                   // 16-byte words per stage and row
    const int wpr = kbw * WPS;                                    // words per row in the slice
    const int words = M * wpr;
    const uint32_t xq = xs.xq + (uint32_t)(warp * xs.wq), xsum = xs.xsum + (uint32_t)(warp * xs.ws);
    const int xrb = xw_row_bytes(M, KB, BITS), xsrb = xsw_row_bytes(M, KB, BITS);
    constexpr int NW = XROOM / 16 / kConsumerThreads;              // words per lane at most
    uint4 v[NW];
    int row[NW];
    // all loads first (one L2 round trip), then the row maxima
#pragma unroll
    for (int u = 0; u < NW; ++u) {
        const int wi = u * 32 + lane;
        row[u] = 0;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (wi < words) {
            const int m = ONE_ROW ? 0 : wi / wpr, r = wi - m * wpr;
            const int kb = r / WPS, iw = r - kb * WPS;
            row[u] = m;
            v[u] = ldg_cg_v4(xg + (size_t)m * ldx + (size_t)(kb * kConsumerWarps + warp) * Gm::kWarpCodes + iw * 8);
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
        if (u * 32 >= words) break;   // uniform over the warp
        const int wi = u * 32 + lane;
        float s_part = 0.f, p_part = 0.f;
        const int m = row[u];
        int em = e[0];
        if (!ONE_ROW) {
#pragma unroll
            for (int mm = 1; mm < MR; ++mm) em = m == mm ? e[mm] : em;
        }
        const int r = wi - m * wpr, kb = r / WPS, iw = r - kb * WPS;
        if (wi < words) {
            const float sc = pow2f(em);
            const float sc16 = sc * 0.0625f;   // 4-bit: codes at bits 4-7 of a byte weigh 16x
            const uint4 a = v[u];
            const float x0 = bf16lo(a.x) * sc, x1 = bf16hi(a.x) * sc, x2 = bf16lo(a.y) * sc, x3 = bf16hi(a.y) * sc;
            const float x4 = bf16lo(a.z) * sc, x5 = bf16hi(a.z) * sc, x6 = bf16lo(a.w) * sc, x7 = bf16hi(a.w) * sc;
            uint32_t p0, p1, p2, p3;
            if (BITS == 4) {
                // fragment registers: (x0, x4), (x1, x5)/16, (x2, x6), (x3, x7)/16
                p0 = f32x2_to_f16x2(x0, x4);
                p1 = f32x2_to_f16x2(bf16hi(a.x) * sc16, bf16hi(a.z) * sc16);
                p2 = f32x2_to_f16x2(x2, x6);
                p3 = f32x2_to_f16x2(bf16hi(a.y) * sc16, bf16hi(a.w) * sc16);
            } else {
                // the chunk is code words 2c, 2c+1 of 8-bit codes: (x0, x2), (x1, x3), (x4, x6), (x5, x7)
                p0 = f32x2_to_f16x2(x0, x2);
                p1 = f32x2_to_f16x2(x1, x3);
                p2 = f32x2_to_f16x2(x4, x6);
                p3 = f32x2_to_f16x2(x5, x7);
            }
            s_part = ((x0 + x1) + (x2 + x3)) + ((x4 + x5) + (x6 + x7));
            p_part = (f16x2_sum(p0) + f16x2_sum(p1)) + (f16x2_sum(p2) + f16x2_sum(p3));
            const int gl = iw >> 3, w8 = iw & 7;
            const uint32_t q = xq + (uint32_t)(m * xrb + kb * (Gm::kGroupsPerWarp * 128) + gl * 128 + (w8 & 1) * 64 +
                                               (w8 >> 1) * 4);
            sts32(q, p0);
            sts32(q + 16, p1);
            sts32(q + 32, p2);
            sts32(q + 48, p3);
        }
        // the 8 words of a group sit in 8 consecutive lanes: fixed-order sums
        s_part += __shfl_xor_sync(0xFFFFFFFFu, s_part, 1);
        p_part += __shfl_xor_sync(0xFFFFFFFFu, p_part, 1);
        s_part += __shfl_xor_sync(0xFFFFFFFFu, s_part, 2);
        p_part += __shfl_xor_sync(0xFFFFFFFFu, p_part, 2);
        s_part += __shfl_xor_sync(0xFFFFFFFFu, s_part, 4);
        p_part += __shfl_xor_sync(0xFFFFFFFFu, p_part, 4);
        if (wi < words && (wi & 7) == 0)
            sts64(xsum + (uint32_t)(m * xsrb + (kb * Gm::kGroupsPerWarp + (iw >> 3)) * 8), s_part, p_part);
    }
    if (ONE_ROW) {
        inv[0] = inv[1] = pow2f(-e[0]);
    } else {
        const int j = lane & 3;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int r0 = 8 * nb + 2 * j < M ? 8 * nb + 2 * j : M - 1;
            const int r1 = 8 * nb + 2 * j + 1 < M ? 8 * nb + 2 * j + 1 : M - 1;
            int e0 = e[0], e1 = e[0];
#pragma unroll
            for (int mm = 1; mm < MR; ++mm) {
                e0 = r0 == mm ? e[mm] : e0;
                e1 = r1 == mm ? e[mm] : e1;
            }
            inv[2 * nb] = pow2f(-e0);
            inv[2 * nb + 1] = pow2f(-e1);
        }
    }
    __syncwarp();   // the region is written before any lane's ldmatrix reads it
}

// Per-thread shared-memory offsets, fixed while one matrix is processed.
struct ConsumerThread {
    uint32_t code[2];   // stage offsets of the code words of row lane/4, groups 2w and 2w+1 (rows +8 at +1024)
    uint32_t sb;        // offset in a scale box of row lane/4's scales of groups 2w, 2w+1 (rows +8 at +512)
    uint32_t xq;        // ldmatrix row address of this warp's first quad in stage 0
    uint32_t xs0, xs1;  // (Xs, X') of this warp's first group in stage 0, x rows of columns 2j and 2j+1
    uint32_t xq1;       // with a second block of 8 columns (x rows 8..15): its ldmatrix row address
    uint32_t xs2, xs3;  // and its (Xs, X') addresses, x rows 8 + 2j and 8 + 2j + 1
};

// K: the codes of the staged x (the matmul's K, or one K pass).
template <int BITS, bool ONE_ROW, int NB = 1>
__device__ __forceinline__ void consumer_init(ConsumerThread &c, int warp, int lane, const XStage &xs, int M_, int K) {
    const int M = ONE_ROW ? 1 : M_;
    using Gm = Geo<BITS>;
    const int gid = lane >> 2, j = lane & 3;
    // code boxes use the 128-byte swizzle: 16-byte chunk c of box row r sits at chunk c ^ (r % 8)
    if (BITS == 4) {
        // words 2j, 2j+1 of groups 2w, 2w+1: 8 bytes per group
        const int c0 = (4 * (warp & 1)) | (j >> 1);
#pragma unroll
        for (int gl = 0; gl < 2; ++gl)
            c.code[gl] = (uint32_t)((warp >> 1) * kBoxBytes + gid * 128 + (((c0 ^ gid) ^ (2 * gl)) << 4) + ((j & 1) << 3));
        // scale boxes (64-byte rows), 64-byte swizzle: chunk c of row r sits at chunk c ^ ((r / 2) % 4)
        c.sb = (uint32_t)(gid * 64 + (((warp >> 2) ^ ((gid >> 1) & 3)) << 4) + ((warp & 3) << 2));
    } else {
        // words 4j..4j+3 of group w: 16 bytes
        const int c0 = 4 * (warp & 1) + j;
        c.code[0] = c.code[1] = (uint32_t)((warp >> 1) * kBoxBytes + gid * 128 + ((c0 ^ gid) << 4));
        // scale boxes (32-byte rows), 32-byte swizzle: chunk bit 0 ^= row bit 2; the word of groups
        // w & ~1 and w | 1
        c.sb = (uint32_t)(gid * 32 + ((((warp >> 3) ^ (gid >> 2)) & 1) << 4) + (((warp >> 1) & 3) << 2));
    }
    const int KB = (K + Gm::kStageCodes - 1) / Gm::kStageCodes;
    const int xr = (lane & 7) < M ? (lane & 7) : M - 1;
    c.xq = xs.xq + (uint32_t)(warp * xs.wq + xr * xw_row_bytes(M, KB, BITS) + (lane >> 3) * 16);
    const int xsrb = xsw_row_bytes(M, KB, BITS);
    const int m0 = 2 * j < M ? 2 * j : M - 1, m1 = 2 * j + 1 < M ? 2 * j + 1 : M - 1;
    c.xs0 = xs.xsum + (uint32_t)(warp * xs.ws + m0 * xsrb);
    c.xs1 = xs.xsum + (uint32_t)(warp * xs.ws + m1 * xsrb);
    if (NB == 2) {
        const int xr1 = 8 + (lane & 7) < M ? 8 + (lane & 7) : M - 1;
        c.xq1 = xs.xq + (uint32_t)(warp * xs.wq + xr1 * xw_row_bytes(M, KB, BITS) + (lane >> 3) * 16);
        const int m2 = 8 + 2 * j < M ? 8 + 2 * j : M - 1, m3 = 8 + 2 * j + 1 < M ? 8 + 2 * j + 1 : M - 1;
        c.xs2 = xs.xsum + (uint32_t)(warp * xs.ws + m2 * xsrb);
        c.xs3 = xs.xsum + (uint32_t)(warp * xs.ws + m3 * xsrb);
    }
}

// acc += scale * (D - 1024 X') + bias * Xs for one group: D = d[h] (the MMA
// accumulators of row block h), scale/bias of rows gid + 8r in s[r], b[r],
// (Xs, X') of the group at xs0 (column 2j) and xs1 (column 2j+1).
template <bool ONE_ROW>
__device__ __forceinline__ void fold_group(const float (&d)[2][4], const float (&sc)[4], const float (&bi)[4],
                                           uint32_t xs0, uint32_t xs1, float (&acc)[2][4]) {
    if (ONE_ROW) {
        const uint2 xv = lds64(xs0);
        const float xsum = __uint_as_float(xv.x), xpr = __uint_as_float(xv.y);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float2 s2 = make_float2(sc[2 * h], sc[2 * h + 1]);
            const float2 b2 = make_float2(bi[2 * h], bi[2 * h + 1]);
            const float2 t = fma2(make_float2(-1024.f, -1024.f), make_float2(xpr, xpr), make_float2(d[h][0], d[h][2]));
            const float2 a = fma2(s2, t, fma2(b2, make_float2(xsum, xsum), make_float2(acc[h][0], acc[h][2])));
            acc[h][0] = a.x;
            acc[h][2] = a.y;
        }
    } else {
        const uint2 xa = lds64(xs0), xb = lds64(xs1);
        const float2 xsum = make_float2(__uint_as_float(xa.x), __uint_as_float(xb.x));
        const float2 xpr = make_float2(__uint_as_float(xa.y), __uint_as_float(xb.y));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const float s = sc[2 * h + rr], b = bi[2 * h + rr];
                const float2 t = fma2(make_float2(-1024.f, -1024.f), xpr, make_float2(d[h][2 * rr], d[h][2 * rr + 1]));
                const float2 a = fma2(make_float2(s, s), t,
                                      fma2(make_float2(b, b), xsum, make_float2(acc[h][2 * rr], acc[h][2 * rr + 1])));
                acc[h][2 * rr] = a.x;
                acc[h][2 * rr + 1] = a.y;
            }
        }
    }
}

// fold_group for one row block (rows gid and gid + 8: scales s0, s1 and
// biases b0, b1), several rows of x: acc += s * (D - 1024 X') + b * Xs.
__device__ __forceinline__ void fold_rows(const float (&d)[4], float s0, float s1, float b0, float b1, uint32_t xs0,
                                          uint32_t xs1, float (&acc)[4]) {
    const uint2 xa = lds64(xs0), xb = lds64(xs1);
    const float2 xsum = make_float2(__uint_as_float(xa.x), __uint_as_float(xb.x));
    const float2 xpr = make_float2(__uint_as_float(xa.y), __uint_as_float(xb.y));
    const float2 t0 = fma2(make_float2(-1024.f, -1024.f), xpr, make_float2(d[0], d[1]));
    const float2 t1 = fma2(make_float2(-1024.f, -1024.f), xpr, make_float2(d[2], d[3]));
    const float2 a0 = fma2(make_float2(s0, s0), t0, fma2(make_float2(b0, b0), xsum, make_float2(acc[0], acc[1])));
    const float2 a1 = fma2(make_float2(s1, s1), t1, fma2(make_float2(b1, b1), xsum, make_float2(acc[2], acc[3])));
    acc[0] = a0.x;
    acc[1] = a0.y;
    acc[2] = a1.x;
    acc[3] = a1.y;
}

// Adds the warp's block of stage `st` (32 rows x 128 bytes of codes; stage
// index kb of the tile) to acc.  acc[h][*] are the MMA accumulator registers
// of row block h: (row, column) = (gid, 2j), (gid, 2j+1), (gid+8, 2j),
// (gid+8, 2j+1).
template <int BITS, bool ONE_ROW>
__device__ __forceinline__ void consume_stage(uint32_t st, int kb, const ConsumerThread &c, float (&acc)[2][4]) {
    using Gm = Geo<BITS>;
    uint32_t sw[4], bw[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        sw[r] = lds32(st + kCodesBytes + c.sb + 8 * Gm::kSBRowBytes * r);
        bw[r] = lds32(st + kCodesBytes + kSBRegion + c.sb + 8 * Gm::kSBRowBytes * r);
    }
    const uint32_t xq = c.xq + (uint32_t)kb * (Gm::kGroupsPerWarp * 128);
    const uint32_t xo = (uint32_t)kb * (Gm::kGroupsPerWarp * 8);
    if (BITS == 4) {
        // every shared-memory load of the stage first, then the arithmetic
        uint2 wrs[2][4];
        uint4 Xs[2][2];
#pragma unroll
        for (int gl = 0; gl < 2; ++gl) {
#pragma unroll
            for (int r = 0; r < 4; ++r) wrs[gl][r] = lds64(st + c.code[gl] + 1024 * r);
#pragma unroll
            for (int i = 0; i < 2; ++i) Xs[gl][i] = ldsm_x4(xq + gl * 128 + i * 64);
        }
#pragma unroll
        for (int gl = 0; gl < 2; ++gl) {
            uint2 wr[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) wr[r] = wrs[gl][r];
            float d[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint4 X = Xs[gl][i];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t wa = i ? wr[2 * h].y : wr[2 * h].x;
                    const uint32_t wb = i ? wr[2 * h + 1].y : wr[2 * h + 1].x;
                    const uint32_t ta = wa >> 8, tb = wb >> 8;
                    if (i == 0)
                        mma_f16_16816_zc(d[h], lo_pair(wa), lo_pair(wb), hi_pair(wa), hi_pair(wb), X.x, X.y);
                    else
                        mma_f16_16816(d[h], lo_pair(wa), lo_pair(wb), hi_pair(wa), hi_pair(wb), X.x, X.y);
                    mma_f16_16816(d[h], lo_pair(ta), lo_pair(tb), hi_pair(ta), hi_pair(tb), X.z, X.w);
                }
            }
            float sc[4], bi[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                sc[r] = gl ? bf16hi(sw[r]) : bf16lo(sw[r]);
                bi[r] = gl ? bf16hi(bw[r]) : bf16lo(bw[r]);
            }
            fold_group<ONE_ROW>(d, sc, bi, c.xs0 + xo + gl * 8, c.xs1 + xo + gl * 8, acc);
        }
    } else {
        // 8-bit: thread j holds words 4j..4j+3 of its rows' group; k-step s of
        // the MMA takes word 4j + s, bytes (0, 2) and (1, 3) as two code pairs
        uint4 wr[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) wr[r] = lds128(st + c.code[0] + 1024 * r);
        float d[2][4];
#pragma unroll
        for (int sp = 0; sp < 2; ++sp) {
            const uint4 X = ldsm_x4(xq + sp * 64);
#pragma unroll
            for (int ss = 0; ss < 2; ++ss) {
                const int s = 2 * sp + ss;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 &A = wr[2 * h], &B = wr[2 * h + 1];
                    const uint32_t wa = s == 0 ? A.x : s == 1 ? A.y : s == 2 ? A.z : A.w;
                    const uint32_t wb = s == 0 ? B.x : s == 1 ? B.y : s == 2 ? B.z : B.w;
                    const uint32_t b0 = ss ? X.z : X.x, b1 = ss ? X.w : X.y;
                    if (s == 0)
                        mma_f16_16816_zc(d[h], byte_pair(wa), byte_pair(wb), byte_pair(wa >> 8), byte_pair(wb >> 8), b0, b1);
                    else
                        mma_f16_16816(d[h], byte_pair(wa), byte_pair(wb), byte_pair(wa >> 8), byte_pair(wb >> 8), b0, b1);
                }
            }
        }
        const int odd = threadIdx.x >> 5 & 1;   // the warp's group is the high half of its scale word
        float sc[4], bi[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            sc[r] = odd ? bf16hi(sw[r]) : bf16lo(sw[r]);
            bi[r] = odd ? bf16hi(bw[r]) : bf16lo(bw[r]);
        }
        fold_group<ONE_ROW>(d, sc, bi, c.xs0 + xo, c.xs1 + xo, acc);
    }
}

// consume_stage for 9..16 rows of x: two blocks of 8 MMA columns (x rows 0..7
// and 8..15).  Each code pair is extracted once and feeds both blocks' MMAs;
// acc[nb] holds block nb.
template <int BITS>
__device__ __forceinline__ void consume_stage2(uint32_t st, int kb, const ConsumerThread &c, float (&acc)[2][2][4]) {
    using Gm = Geo<BITS>;
    const uint32_t sbase = st + kCodesBytes + c.sb;   // scale word of row gid + 8r at + 8 * kSBRowBytes * r
    const uint32_t xo = (uint32_t)kb * (Gm::kGroupsPerWarp * 8);
    const uint32_t xq[2] = {c.xq + (uint32_t)kb * (Gm::kGroupsPerWarp * 128),
                            c.xq1 + (uint32_t)kb * (Gm::kGroupsPerWarp * 128)};
    const uint32_t xsa[2] = {c.xs0 + xo, c.xs2 + xo}, xsb[2] = {c.xs1 + xo, c.xs3 + xo};
    if (BITS == 4) {
        // one row block h at a time, so that only its accumulators (two blocks of
        // columns) are live beside acc: the whole stage's at once spill
#pragma unroll
        for (int gl = 0; gl < 2; ++gl) {
            uint2 wr[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) wr[r] = lds64(st + c.code[gl] + 1024 * r);
            uint4 X[2][2];   // [quad i][column block]
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) X[i][nb] = ldsm_x4(xq[nb] + gl * 128 + i * 64);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float d[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint32_t wa = i ? wr[2 * h].y : wr[2 * h].x;
                    const uint32_t wb = i ? wr[2 * h + 1].y : wr[2 * h + 1].x;
                    const uint32_t ta = wa >> 8, tb = wb >> 8;
                    const uint32_t a0 = lo_pair(wa), a1 = lo_pair(wb), a2 = hi_pair(wa), a3 = hi_pair(wb);
                    const uint32_t b0 = lo_pair(ta), b1 = lo_pair(tb), b2 = hi_pair(ta), b3 = hi_pair(tb);
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb) {
                        if (i == 0)
                            mma_f16_16816_zc(d[nb], a0, a1, a2, a3, X[i][nb].x, X[i][nb].y);
                        else
                            mma_f16_16816(d[nb], a0, a1, a2, a3, X[i][nb].x, X[i][nb].y);
                        mma_f16_16816(d[nb], b0, b1, b2, b3, X[i][nb].z, X[i][nb].w);
                    }
                }
                // this row block's scale and bias words, loaded here rather than
                // held across the stage
                const uint32_t s0 = lds32(sbase + 8 * Gm::kSBRowBytes * (2 * h));
                const uint32_t s1 = lds32(sbase + 8 * Gm::kSBRowBytes * (2 * h + 1));
                const uint32_t b0 = lds32(sbase + kSBRegion + 8 * Gm::kSBRowBytes * (2 * h));
                const uint32_t b1 = lds32(sbase + kSBRegion + 8 * Gm::kSBRowBytes * (2 * h + 1));
#pragma unroll
                for (int nb = 0; nb < 2; ++nb)
                    fold_rows(d[nb], gl ? bf16hi(s0) : bf16lo(s0), gl ? bf16hi(s1) : bf16lo(s1),
                              gl ? bf16hi(b0) : bf16lo(b0), gl ? bf16hi(b1) : bf16lo(b1), xsa[nb] + gl * 8,
                              xsb[nb] + gl * 8, acc[nb][h]);
            }
        }
    } else {
        uint32_t sw[4], bw[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            sw[r] = lds32(sbase + 8 * Gm::kSBRowBytes * r);
            bw[r] = lds32(sbase + kSBRegion + 8 * Gm::kSBRowBytes * r);
        }
        uint4 wr[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) wr[r] = lds128(st + c.code[0] + 1024 * r);
        float d[2][2][4];
#pragma unroll
        for (int sp = 0; sp < 2; ++sp) {
            uint4 X[2];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) X[nb] = ldsm_x4(xq[nb] + sp * 64);
#pragma unroll
            for (int ss = 0; ss < 2; ++ss) {
                const int s = 2 * sp + ss;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 &A = wr[2 * h], &B = wr[2 * h + 1];
                    const uint32_t wa = s == 0 ? A.x : s == 1 ? A.y : s == 2 ? A.z : A.w;
                    const uint32_t wb = s == 0 ? B.x : s == 1 ? B.y : s == 2 ? B.z : B.w;
                    const uint32_t a0 = byte_pair(wa), a1 = byte_pair(wb), a2 = byte_pair(wa >> 8),
                                   a3 = byte_pair(wb >> 8);
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb) {
                        const uint32_t b0 = ss ? X[nb].z : X[nb].x, b1 = ss ? X[nb].w : X[nb].y;
                        if (s == 0)
                            mma_f16_16816_zc(d[nb][h], a0, a1, a2, a3, b0, b1);
                        else
                            mma_f16_16816(d[nb][h], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
        }
        const int odd = threadIdx.x >> 5 & 1;   // the warp's group is the high half of its scale word
        float sc[4], bi[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            sc[r] = odd ? bf16hi(sw[r]) : bf16lo(sw[r]);
            bi[r] = odd ? bf16hi(bw[r]) : bf16lo(bw[r]);
        }
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) fold_group<false>(d[nb], sc, bi, xsa[nb], xsb[nb], acc[nb]);
    }
}

// This warp's partial sums of a tile, times the x scale 2^-e of their column
// (exact: a power of two; inv[c] for column 2j + c, j = lane % 4), into rw =
// its [kRows][M] slice; gid: the tile row (mod 8) of this lane's MMA rows;
// acc is cleared.
template <bool ONE_ROW>
__device__ __forceinline__ void write_partials(float *rw, int M, int lane, int gid, float (&acc)[2][4],
                                               const float (&inv)[2]) {
    const int j = lane & 3;
    if (ONE_ROW) {
        if (j == 0) {  // every column holds x row 0: lanes j > 0 carry copies
            const float sc = inv[0];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                rw[16 * h + gid] = acc[h][0] * sc;
                rw[16 * h + gid + 8] = acc[h][2] * sc;
            }
        }
    } else {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int m = 2 * j + cc;
            if (m < M) {
                const float sc = inv[cc];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) rw[(16 * h + gid + 8 * rr) * M + m] = acc[h][2 * rr + cc] * sc;
            }
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.f;
}

// ---------------------------------------------------------------- end of a tile
//
// Every consumer warp deposits its partial sums of a tile in one of
// red_bufs<ONE_ROW> rotating buffers and moves on to the next tile; a
// dedicated reducer warp adds the sixteen partials of each tile in a fixed
// order and stores y.  The consumers never wait for one another here (a
// buffer is reused only after the reducer has emptied it), and every sum has
// a fixed order, so results do not depend on timing.
// (NB = 2, i.e. 9..16 rows of x: one buffer, whose 32 KB would otherwise crowd out x)
template <bool ONE_ROW, int NB = 1>
__host__ __device__ constexpr int red_bufs() { return ONE_ROW ? 4 : (NB == 2 ? 1 : 2); }
// bytes of the partial-sum buffers: float [bufs][kConsumerWarps][kRows][M]
__host__ __device__ constexpr int red_bytes(int m) {
    return (m == 1 ? 4 : (m > 8 ? 1 : 2)) * kConsumerWarps * kRows * m * 4;
}

struct TileCtx {
    float *red;            // float [bufs][kConsumerWarps][kRows][M]
    uint32_t red_full;     // bufs mbarriers: every warp's sums are in red[b] (count kConsumerWarps)
    uint32_t red_empty;    // bufs mbarriers: red[b] is free again (count 1)
};

// Consumer side, after the last stage of the tcount-th tile of this CTA.
// False on a timeout.
template <bool ONE_ROW>
__device__ __forceinline__ bool deposit_tile(const TileCtx &t, float (&acc)[2][4], int tcount, int M, int warp,
                                             int lane, int gid, const float (&inv)[2], uint64_t timeout_ns,
                                             const volatile int *abort_flag) {
    constexpr int B = red_bufs<ONE_ROW>();
    const int b = tcount % B;
    const int n_out = kRows * M;
    if (tcount >= B && !mbar_wait_for(t.red_empty + 8 * b, (uint32_t)((tcount / B) - 1) & 1u, timeout_ns, abort_flag))
        return false;
    write_partials<ONE_ROW>(t.red + (b * kConsumerWarps + warp) * n_out, M, lane, gid, acc, inv);
    __syncwarp();
    if (lane == 0) mbar_arrive(t.red_full + 8 * b);
    return true;
}

// deposit_tile for two blocks of 8 MMA columns (9..16 rows of x): block nb
// holds x rows 8nb + 2j + c, unscaled by inv[2nb + c].
__device__ __forceinline__ bool deposit_tile2(const TileCtx &t, float (&acc)[2][2][4], int tcount, int M, int warp,
                                              int lane, const float (&inv)[4], uint64_t timeout_ns,
                                              const volatile int *abort_flag) {
    constexpr int B = red_bufs<false, 2>();
    const int b = tcount % B;
    const int n_out = kRows * M;
    if (tcount >= B && !mbar_wait_for(t.red_empty + 8 * b, (uint32_t)((tcount / B) - 1) & 1u, timeout_ns, abort_flag))
        return false;
    float *rw = t.red + (b * kConsumerWarps + warp) * n_out;
    const int gid = lane >> 2, j = lane & 3;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int m = 8 * nb + 2 * j + cc;
            if (m < M) {
                const float sc = inv[2 * nb + cc];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr)
                        rw[(16 * h + gid + 8 * rr) * M + m] = acc[nb][h][2 * rr + cc] * sc;
            }
        }
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int h = 0; h < 2; ++h) acc[nb][h][0] = acc[nb][h][1] = acc[nb][h][2] = acc[nb][h][3] = 0.f;
    __syncwarp();
    if (lane == 0) mbar_arrive(t.red_full + 8 * b);
    return true;
}

// Reducer warp, for the tcount-th tile of this CTA (tile index `tile` of a
// matrix with N rows): adds the (already unscaled) partials in warp order and
// stores y rows tile*kRows .. (bf16, round to nearest even).
//
// When K is walked in several passes (pass `pass` of `passes`), the tile's
// sums of the passes before the last are kept in yacc (float [kRows][M]):
// assigned by the first pass, added to by the next ones, in pass order.
template <bool ONE_ROW, int NB = 1>
__device__ __forceinline__ bool reduce_tile(const TileCtx &t, int tcount, int tile, int M, int N,
                                            __nv_bfloat16 *y, int lane, uint64_t timeout_ns,
                                            const volatile int *abort_flag, float *yacc = nullptr, int pass = 0,
                                            int passes = 1, float yscale = 1.f, int part = 0, int parts = 1) {
    constexpr int B = red_bufs<ONE_ROW, NB>();
    const int b = tcount % B;
    const int n_out = kRows * M;
    // this reducer's share of the outputs: rows [part, part + 1) * kRows / parts of the tile
    const int o0 = part * (kRows / parts) * M, o1 = o0 + (kRows / parts) * M;
    if (!mbar_wait_for(t.red_full + 8 * b, (uint32_t)(tcount / B) & 1u, timeout_ns, abort_flag)) return false;
    const float *rb = t.red + b * kConsumerWarps * n_out;
    if (!ONE_ROW && (M & 3) == 0) {
        // four outputs (one row of W, four rows of x) per lane and step: 16-byte
        // loads and paired adds, the same warp order as below, so the same sums
        for (int idx = o0 + lane * 4; idx < o1; idx += 128) {
            const float4 f0 = *reinterpret_cast<const float4 *>(rb + idx);
            float2 lo = make_float2(f0.x, f0.y), hi = make_float2(f0.z, f0.w);
#pragma unroll
            for (int w = 1; w < kConsumerWarps; ++w) {
                const float4 f = *reinterpret_cast<const float4 *>(rb + w * n_out + idx);
                lo = add2(lo, make_float2(f.x, f.y));
                hi = add2(hi, make_float2(f.z, f.w));
            }
            if (pass > 0) {
                const float4 a = *reinterpret_cast<const float4 *>(yacc + idx);
                lo = add2(make_float2(a.x, a.y), lo);
                hi = add2(make_float2(a.z, a.w), hi);
            }
            const int row = idx / M, m = idx - row * M;
            const int n = tile * kRows + row;
            if (pass + 1 < passes) {
                *reinterpret_cast<float4 *>(yacc + idx) = make_float4(lo.x, lo.y, hi.x, hi.y);
            } else if (n < N) {
                __nv_bfloat16 *yp = y + (int64_t)m * N + n;
                yp[0] = __float2bfloat16_rn(lo.x * yscale);
                yp[N] = __float2bfloat16_rn(lo.y * yscale);
                yp[2 * (int64_t)N] = __float2bfloat16_rn(hi.x * yscale);
                yp[3 * (int64_t)N] = __float2bfloat16_rn(hi.y * yscale);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(t.red_empty + 8 * b);
        return true;
    }
    if (!ONE_ROW && (M & 1) == 0) {
        // two outputs per lane and step (8-byte loads, paired adds), same order
        for (int idx = o0 + lane * 2; idx < o1; idx += 64) {
            float2 v = *reinterpret_cast<const float2 *>(rb + idx);
#pragma unroll
            for (int w = 1; w < kConsumerWarps; ++w) v = add2(v, *reinterpret_cast<const float2 *>(rb + w * n_out + idx));
            if (pass > 0) v = add2(*reinterpret_cast<const float2 *>(yacc + idx), v);
            const int row = idx / M, m = idx - row * M;
            const int n = tile * kRows + row;
            if (pass + 1 < passes) {
                *reinterpret_cast<float2 *>(yacc + idx) = v;
            } else if (n < N) {
                __nv_bfloat16 *yp = y + (int64_t)m * N + n;
                yp[0] = __float2bfloat16_rn(v.x * yscale);
                yp[N] = __float2bfloat16_rn(v.y * yscale);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(t.red_empty + 8 * b);
        return true;
    }
    for (int idx = o0 + lane; idx < o1; idx += 32) {
        const int row = idx / M, m = idx - row * M;
        const int n = tile * kRows + row;
        float v = rb[idx];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) v += rb[w * n_out + idx];
        if (pass > 0) v = yacc[idx] + v;
        if (pass + 1 < passes)
            yacc[idx] = v;
        else if (n < N)
            y[(int64_t)m * N + n] = __float2bfloat16_rn(v * yscale);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(t.red_empty + 8 * b);
    return true;
}

}  // namespace
}  // namespace qmv
}  // namespace aq
