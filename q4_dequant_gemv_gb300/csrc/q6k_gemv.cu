// q6k_gemv.cu -- Q6_K decode GEMV on GB300: y[b] = W x[b] for the other block
// format of Q4_K_M files ("custom quantized GEMV for decode (Q8_0, Q4_K,
// Q6_K)", dotLLM README, News 2026-03 "CUDA GPU backend"; the GGUF Q6_K
// packing is written out in include/q4k.h).
//
// A 210-byte block is only 2-byte aligned inside a row (rows of K/256 blocks
// follow one another), so neither TMA boxes nor 16-byte loads can address it.
// A warp decodes one block of each of its two rows at a time straight from
// global memory (both rows' loads in flight together): lane L takes
// quant bytes ql[4L..4L+3] (two 16-bit loads), i.e. four weights of sub-block
// pair c1 = (L/8)&1 and four of c1+2, the matching four qh bytes, and the two
// int8 scales of those weights.  Per 32-bit word the four 6-bit codes are
// assembled with a few integer ops; each code becomes q - 32 in fp32 by one
// byte permute (2^23 + q) and one exact subtraction; x is read as float4s
// (staged in shared memory when small, else from L1; each load serves both
// rows).  fp32 accumulation, one warp reduction per row; when a matrix has few
// rows, the 8 warps of a CTA split a row pair's blocks and their partial sums
// are added in warp order (deterministic).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "q4k_internal.h"

namespace q4k {
namespace q6 {

constexpr int kBytes = 210;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxB = 16;
constexpr int RPW = 2;             // rows per warp: their loads overlap, x is read once for both
static_assert(RPW == 2, "the kernel addresses exactly two rows per warp (four measured slower)");

__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p)   // 2-byte aligned
{
    return static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(p)));
}

// Persistent CTAs over groups of RPW * kWarps / wpr rows: warp w works on rows
// RPW (w / wpr) .. + RPW - 1 of the group and on the blocks b with b % wpr ==
// w % wpr.  XS: x
// (B x K fp32) is staged in shared memory once per CTA; otherwise it is read
// from global memory (L1).
template <int BMAX, bool XS>
__global__ void __launch_bounds__(kThreads) q6k_gemv_kernel(const uint8_t *__restrict__ W, const float *__restrict__ x,
                                                           float *__restrict__ y, int N, int nb, int B, int wpr,
                                                           int groups)
{
    extern __shared__ __align__(16) float xs[];
    __shared__ float part[kWarps][RPW][BMAX];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows_per_cta = RPW * (kWarps / wpr);
    const int slice = warp % wpr;
    // this lane's share of a block
    const int h = lane >> 4, c1 = (lane >> 3) & 1, l0 = 4 * (lane & 7);
    const int ql_off = 4 * lane;                          // = 64 h + 32 c1 + l0
    const int qh_off = 128 + 32 * h + l0;
    const int sc_off = 192 + 8 * h + 2 * c1 + (l0 >> 4);   // scale of the low-nibble weights; +4 for the high ones
    const int k_lo = 128 * h + 32 * c1 + l0;              // their first weight; +64 for the high ones
    const int K = nb * 256;
    if constexpr (XS) {
        const float4 *src = reinterpret_cast<const float4 *>(x);
        float4 *dst = reinterpret_cast<float4 *>(xs);
        for (int i = threadIdx.x; i < B * K / 4; i += kThreads) dst[i] = __ldg(src + i);
        __syncthreads();
    }
    const float *xv = XS ? xs : x;
    for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const int rowA = grp * rows_per_cta + RPW * (warp / wpr);
        float acc[RPW][BMAX];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int b = 0; b < BMAX; ++b) acc[r][b] = 0.f;
        if (rowA < N) {
            // a missing second row re-reads the first; its sums are never written
            const uint8_t *wrow0 = W + static_cast<size_t>(rowA) * nb * kBytes;
            const uint8_t *wrow1 = (rowA + 1 < N) ? wrow0 + static_cast<size_t>(nb) * kBytes : wrow0;
            for (int blk = slice; blk < nb; blk += wpr) {
                float w_lo[RPW][4], w_hi[RPW][4], s_lo[RPW], s_hi[RPW];
                uint32_t qlv[RPW], qhv[RPW], scv[RPW], dv[RPW];
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    const uint8_t *A = (r ? wrow1 : wrow0) + static_cast<size_t>(blk) * kBytes;
                    qlv[r] = ld_u16(A + ql_off) | (ld_u16(A + ql_off + 2) << 16);
                    qhv[r] = ld_u16(A + qh_off) | (ld_u16(A + qh_off + 2) << 16);
                    scv[r] = static_cast<uint32_t>(__ldg(A + sc_off)) | (static_cast<uint32_t>(__ldg(A + sc_off + 4)) << 8);
                    dv[r] = ld_u16(A + 208);
                }
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(dv[r])));
                    s_lo[r] = d * static_cast<float>(static_cast<int8_t>(scv[r] & 0xFFu));
                    s_hi[r] = d * static_cast<float>(static_cast<int8_t>(scv[r] >> 8));
                    const uint32_t q_lo = (qlv[r] & 0x0F0F0F0Fu) | (((qhv[r] >> (2 * c1)) & 0x03030303u) << 4);
                    const uint32_t q_hi = ((qlv[r] >> 4) & 0x0F0F0F0Fu) | (((qhv[r] >> (2 * c1 + 4)) & 0x03030303u) << 4);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        w_lo[r][j] = __uint_as_float(__byte_perm(q_lo, 0x4B000000u, 0x7440u | j)) - 8388640.0f;
                        w_hi[r][j] = __uint_as_float(__byte_perm(q_hi, 0x4B000000u, 0x7440u | j)) - 8388640.0f;
                    }
                }
                const float *xb = xv + static_cast<size_t>(blk) * 256 + k_lo;
#pragma unroll
                for (int b = 0; b < BMAX; ++b) {
                    if (b >= B) break;
                    float4 xa, xc;
                    if constexpr (XS) {
                        xa = *reinterpret_cast<const float4 *>(xb + static_cast<size_t>(b) * K);
                        xc = *reinterpret_cast<const float4 *>(xb + static_cast<size_t>(b) * K + 64);
                    } else {
                        xa = __ldg(reinterpret_cast<const float4 *>(xb + static_cast<size_t>(b) * K));
                        xc = __ldg(reinterpret_cast<const float4 *>(xb + static_cast<size_t>(b) * K + 64));
                    }
#pragma unroll
                    for (int r = 0; r < RPW; ++r) {
                        float t_lo = w_lo[r][0] * xa.x;
                        t_lo = fmaf(w_lo[r][1], xa.y, t_lo);
                        t_lo = fmaf(w_lo[r][2], xa.z, t_lo);
                        t_lo = fmaf(w_lo[r][3], xa.w, t_lo);
                        float t_hi = w_hi[r][0] * xc.x;
                        t_hi = fmaf(w_hi[r][1], xc.y, t_hi);
                        t_hi = fmaf(w_hi[r][2], xc.z, t_hi);
                        t_hi = fmaf(w_hi[r][3], xc.w, t_hi);
                        acc[r][b] = fmaf(s_lo[r], t_lo, fmaf(s_hi[r], t_hi, acc[r][b]));
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int b = 0; b < BMAX; ++b) {
                if (b >= B) break;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[r][b] += __shfl_xor_sync(0xffffffffu, acc[r][b], o);
                if (lane == 0) part[warp][r][b] = acc[r][b];
            }
        __syncthreads();
        if (static_cast<int>(threadIdx.x) < rows_per_cta * B) {
            const int rr = threadIdx.x / B, b = threadIdx.x - rr * B;   // rr = RPW * (warp row) + r
            const int wr = rr / RPW, r = rr % RPW;
            const int row = grp * rows_per_cta + rr;
            if (row < N) {
                float sum = part[wr * wpr][r][b];
                for (int q = 1; q < wpr; ++q) sum += part[wr * wpr + q][r][b];
                y[static_cast<size_t>(b) * N + row] = sum;
            }
        }
        __syncthreads();   // part[] is rewritten by the next group
    }
}

}  // namespace q6

// Warps per row: enough warps in flight for the GPU (about 48 per SM), at
// most 8 (one CTA) and at most one per block.
static int q6k_warps_per_row(int64_t N, int nb, int sms)
{
    const long long want = static_cast<long long>(sms) * 48;
    int wpr = 1;
    while (wpr < 8 && wpr * 2 <= nb && static_cast<long long>(N) * wpr < want) wpr *= 2;
    return wpr;
}

// Persistent grid: as many CTAs as fit on the GPU at once (occupancy for this
// shared-memory size), at most one per row group.
template <int BMAX, bool XS>
static cudaError_t q6k_launch(const uint8_t *W, const float *x, float *y, int N, int nb, int B, int wpr, int groups,
                              int sms, size_t smem, cudaStream_t s)
{
    auto kern = q6::q6k_gemv_kernel<BMAX, XS>;
    cudaError_t e;
    if (XS) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, q6::kThreads, smem);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(std::min<long long>(groups, static_cast<long long>(sms) * std::max(occ, 1)));
    kern<<<grid, q6::kThreads, smem, s>>>(W, x, y, N, nb, B, wpr, groups);
    return cudaGetLastError();
}

q4k_status q6k_gemv_impl(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream)
{
    if (!x) return Q4K_ERR_INVALID_ARG;
    if ((!W || !y) && N != 0) return Q4K_ERR_INVALID_ARG;
    if (N < 0 || N > 0x7FFFFFFFll || K <= 0 || (K % 256) != 0 || K / 256 >= (1ll << 24)) return Q4K_ERR_INVALID_ARG;
    if (batch < 1 || batch > q6::kMaxB) return Q4K_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) || (reinterpret_cast<uintptr_t>(x) & 15u)) return Q4K_ERR_MISALIGNED;
    int sms = 0;
    const q4k_status st = check_device(&sms);
    if (st != Q4K_OK) return st;
    if (N == 0) return Q4K_OK;
    const int nb = static_cast<int>(K / 256);
    const int wpr = q6k_warps_per_row(N, nb, sms);
    const int rows_per_cta = q6::RPW * (q6::kWarps / wpr);
    const long long groups = (N + rows_per_cta - 1) / rows_per_cta;
    // x staged in shared memory when it is small enough to leave room for six
    // or more CTAs per SM (a larger x there cost more in latency hiding than
    // it saved in loads: measured); persistent CTAs then load it once each
    const size_t xbytes = static_cast<size_t>(batch) * static_cast<size_t>(K) * 4;
    const bool xs = xbytes <= 32 * 1024;
    if (groups > 0x7FFFFFFFll) return Q4K_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t *Wb = static_cast<const uint8_t *>(W);
    const int n = static_cast<int>(N), g = static_cast<int>(groups), gr = sms;
    cudaError_t e;
    if (batch == 1)
        e = xs ? q6k_launch<1, true>(Wb, x, y, n, nb, batch, wpr, g, gr, xbytes, s)
               : q6k_launch<1, false>(Wb, x, y, n, nb, batch, wpr, g, gr, 0, s);
    else if (batch <= 4)
        e = xs ? q6k_launch<4, true>(Wb, x, y, n, nb, batch, wpr, g, gr, xbytes, s)
               : q6k_launch<4, false>(Wb, x, y, n, nb, batch, wpr, g, gr, 0, s);
    else
        e = xs ? q6k_launch<16, true>(Wb, x, y, n, nb, batch, wpr, g, gr, xbytes, s)
               : q6k_launch<16, false>(Wb, x, y, n, nb, batch, wpr, g, gr, 0, s);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4K_ERR_CUDA;
    }
    return Q4K_OK;
}

}  // namespace q4k
