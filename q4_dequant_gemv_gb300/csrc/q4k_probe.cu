// q4k_probe.cu -- read-only HBM streaming probe (q4k_stream_read).
//
// The decode GEMVs only read their weights, so the ceiling they are measured
// against is the rate at which the GPU can stream a buffer from HBM into
// shared memory, not a copy's read+write rate.  This kernel measures that
// ceiling the way the GEMVs stream: one CTA per SM, each reading its own
// contiguous slice with 32 KB bulk asynchronous copies into a 4-deep ring of
// shared memory, L2 evict-first, nothing written back.  (No counterpart on the
// pages: a measurement aid of this library.)

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/q4k.h"
#include "ptx.cuh"
#include "q4k_internal.h"

namespace q4k {
namespace probe {

constexpr int kChunk = 32 * 1024;
constexpr int kDepth = 4;
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ unsigned int g_probe_error = 0;

__global__ void __launch_bounds__(32, 1) stream_read_kernel(const uint8_t *buf, long long per_cta)
{
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t full[kDepth];
    if (threadIdx.x != 0) return;
    const uint8_t *base = buf + per_cta * blockIdx.x;
    const int n = static_cast<int>(per_cta / kChunk);
    for (int i = 0; i < kDepth; ++i) mbar_init(smem_u32(&full[i]), 1);
    fence_barrier_init();
    const uint64_t pol = l2_policy_evict_first();
    int i = 0;
    for (; i < n; ++i) {
        const int slot = i % kDepth;
        if (i >= kDepth &&
            !mbar_wait_bounded(smem_u32(&full[slot]), static_cast<uint32_t>(((i / kDepth) - 1) & 1), kWaitNs)) {
            atomicOr(&g_probe_error, 1u);
            break;
        }
        mbar_arrive_expect_tx(smem_u32(&full[slot]), kChunk);
        bulk_g2s(smem_u32(ring + slot * kChunk), base + static_cast<long long>(i) * kChunk, kChunk,
                 smem_u32(&full[slot]), pol);
    }
    // every copy issued lands before the CTA exits
    for (int j = std::max(0, i - kDepth); j < i; ++j)
        (void)mbar_wait_bounded(smem_u32(&full[j % kDepth]), static_cast<uint32_t>((j / kDepth) & 1), kWaitNs);
}

}  // namespace probe

q4k_status stream_read_impl(const void *buf, int64_t bytes, int64_t *bytes_read, void *stream)
{
    if (!bytes_read) return Q4K_ERR_INVALID_ARG;
    *bytes_read = 0;
    if (bytes < 0 || (bytes > 0 && !buf)) return Q4K_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(buf) & 15u) return Q4K_ERR_MISALIGNED;
    int sms = 0;
    q4k_status st = check_device(&sms);
    if (st != Q4K_OK) return st;
    const long long per_cta = (bytes / sms / probe::kChunk) * probe::kChunk;
    if (per_cta == 0) return Q4K_OK;
    const int smem = probe::kChunk * probe::kDepth;
    if (cudaFuncSetAttribute(probe::stream_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return Q4K_ERR_CUDA;
    }
    probe::stream_read_kernel<<<sms, 32, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(buf), per_cta);
    if (cudaGetLastError() != cudaSuccess) return Q4K_ERR_CUDA;
    *bytes_read = per_cta * sms;
    return Q4K_OK;
}

unsigned int read_probe_error()
{
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, probe::g_probe_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    return v;
}

bool clear_probe_error()
{
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(probe::g_probe_error, &z, sizeof(z)) == cudaSuccess;
}

}  // namespace q4k
