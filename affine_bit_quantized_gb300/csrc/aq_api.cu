// C ABI of libaq: argument validation, kernel choice and the host utilities.
//
// Validation happens before any CUDA runtime call, so a rejected call never
// touches the device (the boundary behaviour asked for by the "MLX CUDA
// Cleanup Plan" page: small wrappers for status handling, no hidden
// fallbacks, no extra copies or synchronization).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include "aq.h"
#include "aq_internal.h"

// Device status word: bounded device-side waits that expire record
// AQ_DEVICE_STATUS_TIMEOUT here; aq_read_device_status() reads and clears it.
__device__ int g_aq_device_status;

namespace {

thread_local char g_last_cuda_error[256] = "";
constexpr int kMaxDevices = 64;
std::atomic<int *> g_status_ptr[kMaxDevices];
constexpr uint64_t kTimeoutNs = 2000000000ull;      // 2 s: far beyond any legitimate wait
constexpr uint64_t kDebugTimeoutNs = 20000000ull;   // 20 ms for the timeout test hook

// Device address of g_aq_device_status on the current device (looked up once
// per device; the first call on a device must not be inside stream capture).
cudaError_t status_ptr(int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int *p = g_status_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_aq_device_status);
        if (e != cudaSuccess) return e;
        g_status_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

aq_status record_cuda(cudaError_t e) {
    if (e == cudaSuccess) return AQ_OK;
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return AQ_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kMaxDim = (int64_t)1 << 30;  // keeps every per-row index inside 32 bits
constexpr int kQmvMaxRows = 16;                // rows of x per weight-streaming pass

// At least `per_sm` 32-row tiles per SM of the current device (per_sm = 0: at
// least 64 tiles).
bool many_tiles(int64_t N, int per_sm = 2) {
    constexpr int kDevices = 64;
    static std::atomic<int> sms[kDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) {
        cudaGetLastError();
        return false;
    }
    int n = sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        sms[dev].store(n, std::memory_order_relaxed);
    }
    return (N + 31) / 32 >= (per_sm > 0 ? per_sm * (int64_t)n : 64);
}

aq_status validate(const void *x, const uint32_t *w, const void *s, const void *b, void *y,
                   int64_t M, int64_t N, int64_t K, int group_size, int bits) {
    if (M < 0 || N < 0 || K < 0) return AQ_ERR_INVALID_ARG;
    if ((bits != 4 && bits != 8) || group_size != 64) return AQ_ERR_UNSUPPORTED;
    if (K % group_size) return AQ_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return AQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return AQ_OK;
    if (!y) return AQ_ERR_INVALID_ARG;
    if (K == 0) return AQ_OK;
    if (!x || !w || !s || !b) return AQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(s, 2) || !aligned(b, 2) || !aligned(y, 2))
        return AQ_ERR_ALIGNMENT;
    if (bits == 8 && (!aligned(s, 16) || !aligned(b, 16))) return AQ_ERR_ALIGNMENT;
    return AQ_OK;
}

// aq_matmul_bf16_ex, with an optional workspace for x converted once on the tensor-core path
aq_status matmul_impl(const void *x, const uint32_t *w_packed, const void *scales, const void *biases, void *y,
                      int64_t M, int64_t N, int64_t K, int group_size, int bits, int kernel, unsigned flags,
                      void *workspace, size_t workspace_bytes, void *stream) {
    if (kernel != AQ_KERNEL_AUTO && kernel != AQ_KERNEL_QMV && kernel != AQ_KERNEL_QMM)
        return AQ_ERR_INVALID_ARG;
    if (flags & ~(unsigned)(AQ_FLAG_PDL | AQ_FLAG_DEBUG_SKIP_COPY)) return AQ_ERR_INVALID_ARG;
    aq_status st = validate(x, w_packed, scales, biases, y, M, N, K, group_size, bits);
    if (st != AQ_OK || M == 0 || N == 0) return st;
    if (kernel == AQ_KERNEL_QMM && K % 512) return AQ_ERR_UNSUPPORTED;   // the tensor-core kernel's K step
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (K == 0) return record_cuda(cudaMemsetAsync(y, 0, (size_t)(M * N) * 2, cs));

    aq::MatmulArgs a;
    a.w = w_packed;
    a.scales = static_cast<const uint16_t *>(scales);
    a.biases = static_cast<const uint16_t *>(biases);
    a.N = N;
    a.K = K;
    a.pdl = (flags & AQ_FLAG_PDL) != 0;
    a.stream = cs;
    a.debug_skip_copy = (flags & AQ_FLAG_DEBUG_SKIP_COPY) != 0;
    a.timeout_ns = a.debug_skip_copy ? kDebugTimeoutNs : kTimeoutNs;
    st = record_cuda(status_ptr(&a.status));
    if (st != AQ_OK) return st;
    a.x = x;
    a.y = y;
    a.M = M;
    a.bits = bits;
    // TMA-fed decode kernel over launches of at most `rows` rows of x (W is
    // streamed once per launch); false when it cannot take this matrix
    auto tma_rows = [&](int64_t rows, aq_status *out) -> bool {
        a.M = rows < M ? rows : M;
        if (!aq::qmv_tma_supported(a)) return false;   // depends on M only through M <= 8
        if (a.debug_skip_copy && M > rows) return false;   // the hook: one launch
        for (int64_t m0 = 0; m0 < M; m0 += rows) {
            a.x = static_cast<const uint16_t *>(x) + m0 * K;
            a.y = static_cast<uint16_t *>(y) + m0 * N;
            a.M = (M - m0) < rows ? (M - m0) : rows;
            *out = record_cuda(aq::launch_qmv_tma(a));
            if (*out != AQ_OK) break;
        }
        return true;
    };
    if (kernel == AQ_KERNEL_QMM || (kernel == AQ_KERNEL_AUTO && M > kQmvMaxRows)) {
        if (workspace && aligned(workspace, 128) && workspace_bytes >= (size_t)(M * K * 2)) a.xf16 = workspace;
        if (aq::qmm_supported(a)) return record_cuda(aq::launch_qmm(a));
        if (kernel == AQ_KERNEL_QMM || a.debug_skip_copy) return AQ_ERR_UNSUPPORTED;
    }
    // 9..16 rows of x where x of all the rows would need K passes (16 rows of
    // K = 4096: 128 KB): one launch of the TMA-fed kernel whose CTA pairs take the
    // two halves of the rows and walk the same tiles together, so W comes from DRAM
    // about once.  4-bit codes: where each half's x fits one pass, over at least one
    // tile per SM (14336 x 4096 at M = 16: 33.1 -> 21.7 us against two launches of 8
    // rows; 4864 x 4096: 18.1 -> 14.6 us against the general kernel, while at 4096 x
    // 4096 the general kernel leads, 12.5 against 14.6 us); where a half needs passes
    // too, over at least two tiles per SM.  8-bit codes: always (against the two
    // column blocks in K passes, 4096 x 4096 at M = 16: 28.6 -> 16.6 us; 1024 x 4096:
    // 26.9 -> 12.7 us; 4096 x 14336, halves in passes: 87.1 -> 47.3 us).
    auto split_launch = [&](aq_status *out) -> bool {
        if (!(M > 8 && M <= kQmvMaxRows && kernel == AQ_KERNEL_AUTO)) return false;
        a.x = x;
        a.y = y;
        a.M = M;
        if (!aq::qmv_tma_supported(a) || aq::qmv_tma_passes(a) == 1) return false;
        a.M = (M + 1) / 2;
        const bool half_one_pass = aq::qmv_tma_passes(a) == 1;
        a.M = M;
        if (!(bits == 8 || (half_one_pass ? many_tiles(N, 1) : many_tiles(N, 2)))) return false;
        a.split_rows = true;
        *out = record_cuda(aq::launch_qmv_tma(a));
        a.split_rows = false;
        return true;
    };
    if (bits == 8) {
        // 8-bit codes: the TMA-fed decode kernel in launches of up to 16 rows of x
        // wherever it applies (K a multiple of 512); else the general kernel below
        st = AQ_OK;
        if (split_launch(&st)) return st;
        if (tma_rows(kQmvMaxRows, &st)) return st;
    }
    if (M <= kQmvMaxRows && kernel != AQ_KERNEL_QMM) {
        st = AQ_OK;
        if (split_launch(&st)) return st;
        a.x = x;
        a.y = y;
        a.M = M;
        // an explicit AQ_KERNEL_QMV takes the TMA-fed kernel wherever it applies; up
        // to 16 rows of x stream W once
        if (aq::qmv_tma_supported(a) &&
            (kernel == AQ_KERNEL_QMV || a.debug_skip_copy || aq::qmv_tma_preferred(a))) {
            st = AQ_OK;
            if (tma_rows(M, &st)) return st;
        }
    }
    if (a.debug_skip_copy) return AQ_ERR_UNSUPPORTED;  // the general kernel has no copy producer
    // Weight-streaming passes over at most 16 rows of x each.
    for (int64_t m0 = 0; m0 < M; m0 += kQmvMaxRows) {
        a.x = static_cast<const uint16_t *>(x) + m0 * K;
        a.y = static_cast<uint16_t *>(y) + m0 * N;
        a.M = (M - m0) < kQmvMaxRows ? (M - m0) : kQmvMaxRows;
        st = record_cuda(aq::launch_qmv(a));
        if (st != AQ_OK) return st;
    }
    return AQ_OK;
}

}  // namespace

extern "C" {

aq_status aq_matmul_bf16_ex(const void *x, const uint32_t *w_packed, const void *scales,
                            const void *biases, void *y, int64_t M, int64_t N, int64_t K,
                            int group_size, int bits, int kernel, unsigned flags, void *stream) {
    return matmul_impl(x, w_packed, scales, biases, y, M, N, K, group_size, bits, kernel, flags, nullptr, 0, stream);
}

size_t aq_matmul_workspace_bytes(int64_t M, int64_t K) {
    if (M <= kQmvMaxRows || K <= 0 || M > kMaxDim || K > kMaxDim) return 0;
    return (size_t)(M * K * 2);
}

aq_status aq_matmul_bf16_ws(const void *x, const uint32_t *w_packed, const void *scales, const void *biases,
                            void *y, int64_t M, int64_t N, int64_t K, int group_size, int bits, void *workspace,
                            size_t workspace_bytes, void *stream) {
    return matmul_impl(x, w_packed, scales, biases, y, M, N, K, group_size, bits, AQ_KERNEL_AUTO, 0u, workspace,
                       workspace_bytes, stream);
}

aq_status aq_matmul_bf16(const void *x, const uint32_t *w_packed, const void *scales,
                         const void *biases, void *y, int64_t M, int64_t N, int64_t K,
                         int group_size, int bits, void *stream) {
    return aq_matmul_bf16_ex(x, w_packed, scales, biases, y, M, N, K, group_size, bits,
                             AQ_KERNEL_AUTO, 0u, stream);
}

// ---------------------------------------------------------------- host utilities

namespace {

// Nearest-even rounding of a double to bf16 by integer arithmetic on its
// significand: keep 8 significant bits (fewer below 2^-126, where bf16 has
// a fixed spacing of 2^-133), round on the dropped bits.
uint16_t bf16_from_double(double v) {
    uint64_t u;
    std::memcpy(&u, &v, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    const uint64_t mag = u & 0x7FFFFFFFFFFFFFFFull;
    const int biased = (int)(mag >> 52);
    if (biased == 0x7FF) return (mag & 0xFFFFFFFFFFFFFull) ? (uint16_t)(sign | 0x7FC0u) : (uint16_t)(sign | 0x7F80u);
    if (biased == 0) return sign;  // zero or a double subnormal, far below half the least bf16
    const int e = biased - 1023;   // |v| = sig * 2^(e - 52), sig in [2^52, 2^53)
    const uint64_t sig = (mag & 0xFFFFFFFFFFFFFull) | (1ull << 52);
    const int unit = e >= -126 ? e - 7 : -133;  // exponent of the bf16 spacing at |v|
    const int drop = 52 + unit - e;             // significand bits below that spacing
    if (drop > 54) return sign;                 // below a quarter of the least spacing
    uint64_t kept = sig >> drop;
    const uint64_t rest = sig & ((1ull << drop) - 1);
    const uint64_t half = 1ull << (drop - 1);
    if (rest > half || (rest == half && (kept & 1))) ++kept;
    const float f = std::ldexp((float)kept, unit);  // exact, or inf on overflow
    uint32_t fb;
    std::memcpy(&fb, &f, sizeof fb);
    return (uint16_t)(sign | (fb >> 16));
}

double double_from_bf16(uint16_t h) {
    const uint32_t fb = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &fb, sizeof f);
    return f;
}

}  // namespace

aq_status aq_pack_ref(const uint8_t *codes, int64_t N, int64_t K, int bits, uint32_t *w_packed) {
    if (bits != 4 && bits != 8) return AQ_ERR_UNSUPPORTED;
    if (N < 0 || K < 0 || K % (32 / bits)) return AQ_ERR_INVALID_ARG;
    if (N * K == 0) return AQ_OK;
    if (!codes || !w_packed) return AQ_ERR_INVALID_ARG;
    const int per = 32 / bits;
    const unsigned limit = 1u << bits;
    for (int64_t i = 0; i < N * K; ++i)
        if (codes[i] >= limit) return AQ_ERR_INVALID_ARG;
    const int64_t nwords = N * K / per;
    for (int64_t wi = 0; wi < nwords; ++wi) {
        uint32_t word = 0;
        const uint8_t *c = codes + wi * per;  // rows are whole words, so words never straddle rows
        for (int p = per - 1; p >= 0; --p) word = (word << bits) | c[p];
        w_packed[wi] = word;
    }
    return AQ_OK;
}

aq_status aq_quantize_ref(const float *w, int64_t N, int64_t K, int group_size, int bits,
                          uint32_t *w_packed, uint16_t *scales_bf16, uint16_t *biases_bf16) {
    if (bits != 4 && bits != 8) return AQ_ERR_UNSUPPORTED;
    if (group_size <= 0 || N < 0 || K <= 0 || K % group_size || K % (32 / bits))
        return AQ_ERR_INVALID_ARG;
    if (N == 0) return AQ_OK;
    if (!w || !w_packed || !scales_bf16 || !biases_bf16) return AQ_ERR_INVALID_ARG;
    const int top = (1 << bits) - 1;
    const int64_t G = K / group_size;
    std::vector<uint8_t> codes((size_t)K);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const float *seg = w + n * K + g * group_size;
            float lo = seg[0], hi = seg[0];
            for (int i = 1; i < group_size; ++i) {
                lo = seg[i] < lo ? seg[i] : lo;
                hi = seg[i] > hi ? seg[i] : hi;
            }
            const uint16_t s16 = bf16_from_double(((double)hi - (double)lo) / (double)top);
            const uint16_t b16 = bf16_from_double((double)lo);
            scales_bf16[n * G + g] = s16;
            biases_bf16[n * G + g] = b16;
            const double s = double_from_bf16(s16), b = double_from_bf16(b16);
            for (int i = 0; i < group_size; ++i) {
                int q = 0;
                if (s != 0.0) {
                    const double t = std::nearbyint(((double)seg[i] - b) / s);
                    q = t < 0.0 ? 0 : (t > (double)top ? top : (int)t);
                }
                codes[(size_t)(g * group_size + i)] = (uint8_t)q;
            }
        }
        aq_status st = aq_pack_ref(codes.data(), 1, K, bits, w_packed + n * (K * bits / 32));
        if (st != AQ_OK) return st;
    }
    return AQ_OK;
}

size_t aq_chain_workspace_bytes(int count) { return aq::chain_workspace_bytes(count); }

aq_status aq_chain_prepare(const aq_matmul_desc *descs, int count, int group_size, int bits, void *workspace,
                           size_t workspace_bytes, aq_chain_plan *plan) {
    cudaError_t e = cudaSuccess;
    aq_status st = aq::chain_prepare(descs, count, group_size, bits, workspace, workspace_bytes, plan, &e);
    if (st == AQ_ERR_CUDA) record_cuda(e);
    return st;
}

aq_status aq_chain_run(const aq_chain_plan *plan, void *stream) {
    if (!plan || plan->count < 0) return AQ_ERR_INVALID_ARG;
    if (plan->count == 0) return AQ_OK;
    if (!plan->workspace) return AQ_ERR_INVALID_ARG;
    int *status = nullptr;
    aq_status st = record_cuda(status_ptr(&status));
    if (st != AQ_OK) return st;
    return record_cuda(aq::chain_run(plan, kTimeoutNs, status, static_cast<cudaStream_t>(stream)));
}

aq_status aq_chain_run_static(const aq_matmul_desc *descs, int count, int group_size, int bits, void *stream) {
    if (count > aq::chain_static_max()) return AQ_ERR_INVALID_ARG;
    int *status = nullptr;
    if (count > 0) {
        aq_status st = record_cuda(status_ptr(&status));
        if (st != AQ_OK) return st;
    }
    cudaError_t e = cudaSuccess;
    aq_status st = aq::chain_run_static(descs, count, group_size, bits, kTimeoutNs, status,
                                        static_cast<cudaStream_t>(stream), &e);
    if (st == AQ_ERR_CUDA) record_cuda(e);
    return st;
}

const char *aq_status_string(aq_status status) {
    switch (status) {
    case AQ_OK: return "AQ_OK";
    case AQ_ERR_INVALID_ARG: return "AQ_ERR_INVALID_ARG";
    case AQ_ERR_UNSUPPORTED: return "AQ_ERR_UNSUPPORTED";
    case AQ_ERR_ALIGNMENT: return "AQ_ERR_ALIGNMENT";
    case AQ_ERR_CUDA: return "AQ_ERR_CUDA";
    case AQ_ERR_TIMEOUT: return "AQ_ERR_TIMEOUT";
    case AQ_ERR_BAD_INDEX: return "AQ_ERR_BAD_INDEX";
    }
    return "AQ_ERR_UNKNOWN";
}

const char *aq_last_cuda_error(void) { return g_last_cuda_error; }

aq_status aq_read_device_status(void *stream) {
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    aq_status st = record_cuda(cudaStreamSynchronize(cs));
    if (st != AQ_OK) return st;
    int *p = nullptr;
    st = record_cuda(status_ptr(&p));
    if (st != AQ_OK) return st;
    int v = 0;
    st = record_cuda(cudaMemcpyFromSymbolAsync(&v, g_aq_device_status, sizeof v, 0, cudaMemcpyDeviceToHost, cs));
    if (st != AQ_OK) return st;
    const int zero = 0;
    st = record_cuda(cudaMemcpyToSymbolAsync(g_aq_device_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, cs));
    if (st != AQ_OK) return st;
    st = record_cuda(cudaStreamSynchronize(cs));
    if (st != AQ_OK) return st;
    if (v == aq::AQ_DEVICE_STATUS_TIMEOUT) return AQ_ERR_TIMEOUT;
    if (v == aq::AQ_DEVICE_STATUS_BAD_INDEX) return AQ_ERR_BAD_INDEX;
    return AQ_OK;
}

size_t aq_gather_qmm_workspace_bytes(int64_t R, int64_t K, int64_t E) {
    if (R < 0 || K < 0 || E < 0 || R > kMaxDim || K > kMaxDim || E > aq::kMaxExperts) return 0;
    return aq::gather_workspace_bytes(R, K, E);
}

aq_status aq_gather_qmm_bf16(const void *x, const uint32_t *w_packed, const void *scales, const void *biases,
                             const int32_t *lhs_indices, const int32_t *rhs_indices, void *y, int64_t R, int64_t T,
                             int64_t N, int64_t K, int64_t E, int group_size, int bits, void *workspace,
                             size_t workspace_bytes, void *stream) {
    if ((bits != 4 && bits != 8) || group_size != 64) return AQ_ERR_UNSUPPORTED;
    if (R < 0 || T < 1 || N < 1 || K < 1 || E < 1 || E > aq::kMaxExperts) return AQ_ERR_INVALID_ARG;
    if (R > kMaxDim || T > kMaxDim || N > kMaxDim || K > kMaxDim || E * N > kMaxDim) return AQ_ERR_INVALID_ARG;
    if (K % group_size) return AQ_ERR_INVALID_ARG;
    if (K % 512) return AQ_ERR_UNSUPPORTED;   // the tensor-core kernel's K step
    if (R == 0) return AQ_OK;
    if (!x || !w_packed || !scales || !biases || !lhs_indices || !rhs_indices || !y || !workspace)
        return AQ_ERR_INVALID_ARG;
    if (workspace_bytes < aq::gather_workspace_bytes(R, K, E)) return AQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w_packed, 16) || !aligned(scales, 16) || !aligned(biases, 16) ||
        !aligned(lhs_indices, 4) || !aligned(rhs_indices, 4) || !aligned(y, 2) || !aligned(workspace, 128))
        return AQ_ERR_ALIGNMENT;
    aq::GatherArgs g;
    g.x = x;
    g.w = w_packed;
    g.scales = static_cast<const uint16_t *>(scales);
    g.biases = static_cast<const uint16_t *>(biases);
    g.lhs = lhs_indices;
    g.rhs = rhs_indices;
    g.y = y;
    g.R = R;
    g.T = T;
    g.N = N;
    g.K = K;
    g.E = E;
    g.bits = bits;
    g.workspace = workspace;
    g.stream = static_cast<cudaStream_t>(stream);
    g.timeout_ns = kTimeoutNs;
    aq_status st = record_cuda(status_ptr(&g.status));
    if (st != AQ_OK) return st;
    return record_cuda(aq::launch_gather_qmm(g));
}

aq_status aq_matmul_nvfp4_bf16(const void *x, const uint32_t *w_packed, const uint8_t *scales_e4m3,
                               float global_scale, void *y, int64_t M, int64_t N, int64_t K, unsigned flags,
                               void *stream) {
    if (flags & ~(unsigned)AQ_FLAG_PDL) return AQ_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || K % 16) return AQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return AQ_OK;
    if (K == 0 || K % 256 || K > 32768) return AQ_ERR_UNSUPPORTED;
    if (!x || !w_packed || !scales_e4m3 || !y) return AQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w_packed, 16) || !aligned(scales_e4m3, 16) || !aligned(y, 2))
        return AQ_ERR_ALIGNMENT;
    aq::Nvfp4Args a;
    a.x = x;
    a.w = w_packed;
    a.scales = scales_e4m3;
    a.global_scale = global_scale;
    a.y = y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.pdl = (flags & AQ_FLAG_PDL) != 0;
    a.stream = static_cast<cudaStream_t>(stream);
    a.timeout_ns = kTimeoutNs;
    aq_status st = record_cuda(status_ptr(&a.status));
    if (st != AQ_OK) return st;
    // each CTA takes up to 8 rows whose x fits the kernel's 64 KB staging room; one
    // launch takes up to 8 such row blocks, on groups of CTAs that walk the same
    // tiles together, so W comes from DRAM about once per launch
    const int64_t rows = std::min<int64_t>(8, 32768 / K), per_launch = 8 * rows;
    a.rows = (int)rows;
    for (int64_t m0 = 0; m0 < M; m0 += per_launch) {
        a.x = static_cast<const uint16_t *>(x) + m0 * K;
        a.y = static_cast<uint16_t *>(y) + m0 * N;
        a.M = (M - m0) < per_launch ? (M - m0) : per_launch;
        st = record_cuda(aq::launch_nvfp4_qmv(a));
        if (st != AQ_OK) return st;
    }
    return AQ_OK;
}

aq_status aq_read_probe(const void *buf, size_t bytes, void *stream) {
    if (!buf || bytes < 16384) return AQ_ERR_INVALID_ARG;
    if (!aligned(buf, 16)) return AQ_ERR_ALIGNMENT;
    int *status = nullptr;
    aq_status st = record_cuda(status_ptr(&status));
    if (st != AQ_OK) return st;
    return record_cuda(aq::launch_read_probe(buf, bytes, kTimeoutNs, status, static_cast<cudaStream_t>(stream)));
}

int aq_version(void) { return 200; }

}  // extern "C"
