// Read-only stream probe: the HBM read ceiling that the decode kernels'
// roofline fractions are also reported against.
//
// The decode kernels stream packed weights into shared memory with the Tensor
// Memory Accelerator and read nothing else of size, so their ceiling is the
// rate at which TMA bulk copies can read device memory, not a copy's
// read-plus-write rate.  This kernel measures that rate with the same
// mechanism and no arithmetic: one persistent CTA per SM streams its share of
// a buffer through a ring of shared-memory slots with cp.async.bulk, keeping
// kSlots copies in flight.  Nothing reads the slots; the copies are real
// memory reads all the same.  Every wait is bounded like the decode kernels'.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "aq_internal.h"
#include "aq_ptx.cuh"

namespace aq {
namespace {

using namespace dev;

constexpr int kChunk = 16384;   // bytes per bulk copy
constexpr int kSlots = 12;      // copies in flight per SM (192 KB)
constexpr int kProbeSmem = kSlots * kChunk + kSlots * 8 + 1024;

__global__ void __launch_bounds__(32, 1)
read_probe_kernel(const uint8_t *__restrict__ buf, long long chunks, unsigned long long timeout_ns, int *status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    const uint32_t bars = base + kSlots * kChunk;
    if (threadIdx.x != 0) return;
    for (int s = 0; s < kSlots; ++s) mbar_init(bars + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // a contiguous share of the chunks per CTA
    const long long per = (chunks + gridDim.x - 1) / gridDim.x;
    const long long c0 = (long long)blockIdx.x * per;
    const long long c1 = c0 + per < chunks ? c0 + per : chunks;
    const uint64_t deadline = global_timer() + timeout_ns;
    long long issued = 0;
    bool ok = true;
    for (long long c = c0; ok && c < c1; ++c, ++issued) {
        const int slot = (int)(issued % kSlots);
        if (issued >= kSlots) {   // the slot's previous copy has landed
            const uint32_t parity = (uint32_t)(((issued / kSlots) - 1) & 1);
            while (!mbar_try_wait(bars + 8 * slot, parity)) {
                if (global_timer() > deadline) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
        }
        mbar_expect_tx(bars + 8 * slot, kChunk);
        bulk_load(base + slot * kChunk, buf + c * kChunk, kChunk, bars + 8 * slot);
    }
    // every copy lands before the CTA exits (bounded)
    const uint64_t drain = global_timer() + timeout_ns;
    for (long long it = issued > kSlots ? issued - kSlots : 0; it < issued; ++it)
        while (!mbar_try_wait(bars + 8 * (int)(it % kSlots), (uint32_t)((it / kSlots) & 1)) && global_timer() < drain) {
        }
    if (!ok) atomicExch(status, (int)AQ_DEVICE_STATUS_TIMEOUT);
}

std::atomic<int> g_probe_attr[64];

}  // namespace

cudaError_t launch_read_probe(const void *buf, size_t bytes, uint64_t timeout_ns, int *status, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (!g_probe_attr[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(read_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
        if (e != cudaSuccess) return e;
        g_probe_attr[dev].store(1, std::memory_order_release);
    }
    const long long chunks = (long long)(bytes / kChunk);
    read_probe_kernel<<<sms, 32, kProbeSmem, stream>>>(static_cast<const uint8_t *>(buf), chunks,
                                                        (unsigned long long)timeout_ns, status);
    return cudaGetLastError();
}

}  // namespace aq
