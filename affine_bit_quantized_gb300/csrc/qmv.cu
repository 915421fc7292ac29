// Weight-streaming kernel for y = x . dequant(W)^T with 1..16 rows of x.
//
// Decode is bound by streaming the packed weights from memory ("epic: CUDA
// (MLX backend) prefill and decode acceleration program", Diagnosis table and
// its first consequence; "gemma-4 decode carries ~44 ms/token ...", re-scope
// paragraph).  The kernel therefore reads every code, scale and bias exactly
// once and keeps the arithmetic per code small enough for the SMs to keep up
// with HBM.
//
// Arithmetic (fp32 accumulation, folded per group of 64):
//   D[n,m,g] = sum_{k in g} (128 + q[n,k]) * x[m,k]        (tensor core, fp32)
//   X[m,g]   = sum_{k in g} x[m,k]                          (same MMA, ones row)
//   y[m,n]   = sum_g scale[n,g] * D[n,m,g] + (bias[n,g] - 128 * scale[n,g]) * X[m,g]
// which equals sum_k x[m,k] * (scale*q + bias) up to fp32 rounding.
//
// Mapping: the dequantization-free products run on mma.sync m16n8k16 (bf16 in,
// fp32 out) with the weights as the 16-row A operand and x as the 8-column B
// operand.  A code q becomes the exact bf16 value 128 + q by OR-ing the nibble
// into the mantissa of 128.0 (bf16 0x4300), two codes per 32-bit register, so
// converting a code costs about one instruction and the MMA does the multiply
// and the adds.  Because a dot product does not care about the order of k,
// the MMA's k-slots are mapped onto adjacent code pairs so that the B fragment
// is x in its natural layout.  MMA row 15 carries ones, which yields the
// per-group sums of x in the same instruction; a tile therefore covers 15
// weight rows.
//
// 8-bit codes (the general path for K that the TMA-fed kernels do not take,
// i.e. K not a multiple of 512): a code q = 16 h + l does not fit the 8-bit
// significand of bf16 as 128 + q, so each code pair goes through the MMA twice,
// as 128 + l and as 128 + h (one OR each), and the fold becomes
//   y[m,n] = sum_g scale * (D_l + 16 D_h) + (bias - 17 * 128 * scale) * X.
//
// Decomposition: one CTA per 15-row tile; its warps split K into chunks of
// 512 codes (8 groups; 4 groups for 8-bit codes), each warp first issuing all
// loads of its chunk (16 code loads of 8 bytes per thread for 4-bit codes, 8
// of 16 bytes for 8-bit) and only then waiting for the preceding kernel
// (programmatic dependent launch) before reading x.  Partial sums are combined
// across warps in shared memory in a fixed order, so results are
// deterministic.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include "aq_internal.h"

namespace aq {
namespace {

constexpr int kTileRows = 15;             // weight rows per CTA; MMA row 15 carries ones
template <int BITS>
__host__ __device__ constexpr int chunk_groups() { return BITS == 4 ? 8 : 4; }   // groups of 64 codes per warp chunk
constexpr int kMaxWarps = 8;
constexpr uint32_t kOnes = 0x3F803F80u;   // bf16x2 (1.0, 1.0)
constexpr uint32_t kMagic = 0x43004300u;  // bf16x2 (128.0, 128.0)

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// bf16x2 (128 + q[2b], 128 + q[2b+1]) from word w (and w4 = w >> 4).
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t w4, int b) {
    const uint32_t sel = (uint32_t)b | ((uint32_t)b << 4) | ((uint32_t)(4 + b) << 8) | ((uint32_t)(4 + b) << 12);
    return (__byte_perm(w, w4, sel) & 0x000F000Fu) | kMagic;
}

// 8-bit codes: bf16x2 (128 + v[2b], 128 + v[2b+1]) of the low nibbles v of
// bytes 2b and 2b+1 of w (pass w >> 4 for the high nibbles).
__device__ __forceinline__ uint32_t nibble_pair8(uint32_t w, int b) {
    const uint32_t sel = (uint32_t)(2 * b) | ((uint32_t)(2 * b + 1) << 8);
    return (__byte_perm(w, 0u, sel) & 0x000F000Fu) | kMagic;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// MT = number of 8-column MMA tiles of x rows (1: M <= 8, 2: M <= 16); BITS:
// code width (4 or 8).
template <int MT, int BITS>
__global__ void __launch_bounds__(kMaxWarps * 32)
qmv_kernel(const __nv_bfloat16 *__restrict__ x, const uint32_t *__restrict__ w,
           const uint16_t *__restrict__ sc, const uint16_t *__restrict__ bi,
           __nv_bfloat16 *__restrict__ y, int M, int N, int K) {
    __shared__ float red[kMaxWarps][16][8 * MT];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int gid = lane >> 2;  // MMA group: A rows gid and gid+8, B/D column gid
    const int j = lane & 3;     // thread in group: k-slot pair
    const int64_t n0 = (int64_t)blockIdx.x * kTileRows;
    const int G = K >> 6;
    const int64_t words = (int64_t)K * BITS / 32;   // code words per row
    constexpr int kChunkGroups = chunk_groups<BITS>();
    using CodeVec = typename std::conditional<BITS == 4, uint2, uint4>::type;   // a lane's codes of a group
    const bool ones_lane = (gid == 7);  // its second A row is tile row 15: the ones row
    const int64_t r0 = n0 + gid, r1 = n0 + gid + 8;
    const bool v0 = r0 < N;
    const bool v1 = !ones_lane && r1 < N;

    griddep_launch();

    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;

    const int nchunks = (G + kChunkGroups - 1) / kChunkGroups;
    for (int c = warp; c < nchunks; c += nwarps) {
        const int g0 = c * kChunkGroups;
        CodeVec q0[kChunkGroups], q1[kChunkGroups];
        uint32_t sb0[kChunkGroups], sb1[kChunkGroups];  // scale bits | bias bits << 16
#pragma unroll
        for (int gi = 0; gi < kChunkGroups; ++gi) {
            const int g = g0 + gi;
            const bool ok = g < G;
            q0[gi] = CodeVec{};
            q1[gi] = CodeVec{};
            sb0[gi] = 0u;
            sb1[gi] = 0u;
            // the lane's words of the group: 2j, 2j+1 of 8 (4-bit), 4j .. 4j+3 of 16 (8-bit)
            constexpr int WPG = 2 * BITS;   // words per group
            constexpr int WPL = WPG / 4;    // words per lane
            if (ok && v0) {
                q0[gi] = __ldcs(reinterpret_cast<const CodeVec *>(w + r0 * words + g * WPG + WPL * j));
                sb0[gi] = (uint32_t)__ldcs(sc + r0 * G + g) | ((uint32_t)__ldcs(bi + r0 * G + g) << 16);
            }
            if (ok && v1) {
                q1[gi] = __ldcs(reinterpret_cast<const CodeVec *>(w + r1 * words + g * WPG + WPL * j));
                sb1[gi] = (uint32_t)__ldcs(sc + r1 * G + g) | ((uint32_t)__ldcs(bi + r1 * G + g) << 16);
            }
        }
        // x may be produced by the preceding kernel: wait for it only now.
        griddep_wait();
#pragma unroll
        for (int gi = 0; gi < kChunkGroups; ++gi) {
            const int g = g0 + gi;
            if (g >= G) break;
            float d[MT][4];
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) d[t][e] = 0.f;
            float dh[MT][4];   // 8-bit codes: the high nibbles' products
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) dh[t][e] = 0.f;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                // the 8 consecutive k of x this step covers: the lane's word 2j + i
                // (4-bit), or its words 4j + 2i and 4j + 2i + 1 (8-bit)
                const int kw = BITS == 4 ? (g * 8 + 2 * j + i) * 8 : g * 64 + 16 * j + 8 * i;
                uint4 X[MT];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const int m = gid + 8 * t;
                    X[t] = make_uint4(0u, 0u, 0u, 0u);
                    if (m < M) X[t] = __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)m * K + kw));
                }
                if constexpr (BITS == 4) {
                    const uint32_t wa = i ? q0[gi].y : q0[gi].x;
                    const uint32_t wb = i ? q1[gi].y : q1[gi].x;
                    const uint32_t wa4 = wa >> 4, wb4 = wb >> 4;
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const uint32_t a0 = code_pair(wa, wa4, 2 * s);
                        const uint32_t a2 = code_pair(wa, wa4, 2 * s + 1);
                        const uint32_t a1 = ones_lane ? kOnes : code_pair(wb, wb4, 2 * s);
                        const uint32_t a3 = ones_lane ? kOnes : code_pair(wb, wb4, 2 * s + 1);
#pragma unroll
                        for (int t = 0; t < MT; ++t)
                            mma_bf16_16816(d[t], a0, a1, a2, a3, s ? X[t].z : X[t].x, s ? X[t].w : X[t].y);
                    }
                } else {
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        // word 4j + 2i + s: codes at k = kw + 4s .. kw + 4s + 3 (slots 2j, 2j+1, 2j+8, 2j+9)
                        const uint32_t wa = i ? (s ? q0[gi].w : q0[gi].z) : (s ? q0[gi].y : q0[gi].x);
                        const uint32_t wb = i ? (s ? q1[gi].w : q1[gi].z) : (s ? q1[gi].y : q1[gi].x);
#pragma unroll
                        for (int hn = 0; hn < 2; ++hn) {
                            const uint32_t va = hn ? wa >> 4 : wa, vb = hn ? wb >> 4 : wb;
                            const uint32_t a0 = nibble_pair8(va, 0);
                            const uint32_t a2 = nibble_pair8(va, 1);
                            const uint32_t a1 = ones_lane ? kOnes : nibble_pair8(vb, 0);
                            const uint32_t a3 = ones_lane ? kOnes : nibble_pair8(vb, 1);
#pragma unroll
                            for (int t = 0; t < MT; ++t)
                                mma_bf16_16816(hn ? dh[t] : d[t], a0, a1, a2, a3, s ? X[t].z : X[t].x,
                                               s ? X[t].w : X[t].y);
                        }
                    }
                }
            }
            if constexpr (BITS == 8) {
                // D = D_l + 16 D_h; the ones row of D_l alone gives X
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    d[t][0] = fmaf(16.f, dh[t][0], d[t][0]);
                    d[t][1] = fmaf(16.f, dh[t][1], d[t][1]);
                    if (!ones_lane) {
                        d[t][2] = fmaf(16.f, dh[t][2], d[t][2]);
                        d[t][3] = fmaf(16.f, dh[t][3], d[t][3]);
                    }
                }
            }
            // fold: acc += scale * D + (bias - c * scale) * X, c = 128 (4-bit) or 17 * 128 (8-bit)
            constexpr float kOffset = BITS == 4 ? -128.f : -2176.f;
            const float s0 = bf16_bits_to_float(sb0[gi] & 0xFFFFu);
            const float s1 = bf16_bits_to_float(sb1[gi] & 0xFFFFu);
            const float p0 = fmaf(kOffset, s0, bf16_bits_to_float(sb0[gi] >> 16));
            const float p1 = fmaf(kOffset, s1, bf16_bits_to_float(sb1[gi] >> 16));
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const float xs0 = __shfl_sync(0xFFFFFFFFu, d[t][2], 28 + j);
                const float xs1 = __shfl_sync(0xFFFFFFFFu, d[t][3], 28 + j);
                acc[t][0] = fmaf(s0, d[t][0], fmaf(p0, xs0, acc[t][0]));
                acc[t][1] = fmaf(s0, d[t][1], fmaf(p0, xs1, acc[t][1]));
                acc[t][2] = fmaf(s1, d[t][2], fmaf(p1, xs0, acc[t][2]));
                acc[t][3] = fmaf(s1, d[t][3], fmaf(p1, xs1, acc[t][3]));
            }
        }
    }
    griddep_wait();  // y may still be read by the preceding kernel

#pragma unroll
    for (int t = 0; t < MT; ++t) {
        red[warp][gid][8 * t + 2 * j] = acc[t][0];
        red[warp][gid][8 * t + 2 * j + 1] = acc[t][1];
        red[warp][gid + 8][8 * t + 2 * j] = acc[t][2];
        red[warp][gid + 8][8 * t + 2 * j + 1] = acc[t][3];
    }
    __syncthreads();
    const int Mc = M < 8 * MT ? M : 8 * MT;
    for (int idx = threadIdx.x; idx < kTileRows * Mc; idx += blockDim.x) {
        const int m = idx / kTileRows;
        const int row = idx - m * kTileRows;
        const int64_t n = n0 + row;
        if (n < N) {
            float v = red[0][row][m];
            for (int ww = 1; ww < nwarps; ++ww) v += red[ww][row][m];
            y[(int64_t)m * N + n] = __float2bfloat16_rn(v);
        }
    }
}

}  // namespace

cudaError_t launch_qmv(const MatmulArgs &a) {
    const int G = (int)(a.K / 64);
    const int cg = a.bits == 8 ? chunk_groups<8>() : chunk_groups<4>();
    const int nchunks = (G + cg - 1) / cg;
    const int nwarps = std::min(kMaxWarps, nchunks);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.N + kTileRows - 1) / kTileRows));
    cfg.blockDim = dim3(32 * nwarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    const auto *x = static_cast<const __nv_bfloat16 *>(a.x);
    auto *y = static_cast<__nv_bfloat16 *>(a.y);
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K;
    auto kern = a.bits == 8 ? (a.M <= 8 ? qmv_kernel<1, 8> : qmv_kernel<2, 8>)
                            : (a.M <= 8 ? qmv_kernel<1, 4> : qmv_kernel<2, 4>);
    return cudaLaunchKernelEx(&cfg, kern, x, a.w, a.scales, a.biases, y, M, N, K);
}

}  // namespace aq
