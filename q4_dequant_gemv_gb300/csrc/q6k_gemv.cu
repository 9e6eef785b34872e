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

#include "ptx.cuh"
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
                                                           float *__restrict__ y, int N, int ldy, int nb, int B,
                                                           int wpr, int groups)
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
                y[static_cast<size_t>(b) * ldy + row] = sum;
            }
        }
        __syncthreads();   // part[] is rewritten by the next group
    }
}


// ---------------------------------------------------------------------------
// Staged variant, integer inner product (batch <= 4).
//
// Tiles of 8 RW rows, each streamed through shared memory in K-slices (one
// bulk async copy per row and slice, its range rounded out to 16-byte
// boundaries, so the row's first block starts at an even offset inside the
// stage); warp w works on rows w, w + 8, ... of the tile and loads its x
// parts once per block for all of them.  Batch 1 takes RW = 2 in two 48 KB
// stages (two CTAs per SM): the shared-memory load pipe bounds this kernel,
// and the x loads, shared by two rows, are half of its wavefronts (LM head
// 150 -> 125 us against RW = 1 in three 28 KB stages, which batch 2-4 keep).  x is
// converted once per CTA, block by block, into two int8 parts
// (x ~ (a/32258)(254 xh + xl), a = the block's max |x|, rounding to nearest
// even), laid out so that lane L finds the parts of its eight x values in one
// 16-byte word, with the exact int32 sums of each four of them beside.  Each
// lane then forms q (0..63) of its four low and four high weights as packed
// bytes and takes the dot products with dp4a: per scale group
// T = 254 (q . xh) + (q . xl) - 32 X4 is the exact integer sum of (q - 32) x
// in units of the block's step, and sc_lo T_lo + sc_hi T_hi stays exact in
// int32 (|.| < 1.1e9); y += (d u) p (that sum), with u p the block's step.
// (The float path, one fp32 FMA per weight, was instruction-bound.)
// Persistent CTAs over the tiles; the last warp to finish a stage issues the
// stage ST ahead into it.  Every wait is bounded: on a timeout the CTA
// flags g_q6k_error, keeps walking its schedule without waiting, and waits
// (bounded) for its copies in flight before it exits.
// ---------------------------------------------------------------------------
// staging of the batch-1 and the batch-2..4 kernels: rows per warp, stages,
// stage size target
constexpr int kRW1 = 2, kStages1 = 2, kStageKB1 = 48;
constexpr int kRW4 = 1, kStages4 = 3, kStageKB4 = 28;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr int kXItemBytes = 32 * 16 + 32 * 8;      // int8 parts + four-value sums of one (batch row, block)

__device__ unsigned int g_q6k_error = 0;   // bit 0: a bounded wait of the staged kernel timed out

__device__ __forceinline__ uint32_t lds_u16(const uint8_t *p) { return *reinterpret_cast<const unsigned short *>(p); }

// Row pitch of a stage for slices of sb blocks: the slice plus up to 15 bytes
// of rounding on each side, a multiple of 16.
__host__ __device__ inline int q6_pitch(int sb) { return ((sb * kBytes + 30 + 15) / 16) * 16; }

// One (batch row, block) of x for the integer path, by one warp: lane L holds
// x[k_lo .. k_lo + 3] (v0) and x[k_lo + 64 .. + 67] (v1) of the block.
// Writes {xh(v0), xh(v1), xl(v0), xl(v1)} as packed int8 to xq[L], -32 times
// the exact sums 254 xh + xl of each four to x4[L] (the q - 32 offset of the
// weights), and returns {u, p}: x ~ u p (254 xh + xl).  Below 2^-64 the max is scaled by 2^64 first (exact), so that u
// stays normal; p = 2^-64 then.  A block whose max is zero or not finite gets
// zero parts and u = 0 (zero) or u = max (inf/NaN propagate).
__device__ __forceinline__ float2 q6_x_item(float4 v0, float4 v1, int lane, uint4 *xq, int2 *x4)
{
    uint32_t m = 0u;
    m = max(m, max(max(__float_as_uint(fabsf(v0.x)), __float_as_uint(fabsf(v0.y))),
                   max(__float_as_uint(fabsf(v0.z)), __float_as_uint(fabsf(v0.w)))));
    m = max(m, max(max(__float_as_uint(fabsf(v1.x)), __float_as_uint(fabsf(v1.y))),
                   max(__float_as_uint(fabsf(v1.z)), __float_as_uint(fabsf(v1.w)))));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float amax = __uint_as_float(m);
    const bool ok = m != 0u && m < 0x7F800000u;
    const float pre = (m < 0x1F800000u) ? 0x1p64f : 1.0f;
    const float inv = ok ? 127.0f / (amax * pre) : 0.0f;
    constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23: adding it rounds to an integer
    constexpr uint32_t kMagicBits = 0x4B400000u;
    uint32_t hw[2], lw[2];
    int sums[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const float4 w = h2 ? v1 : v0;
        const float e[4] = {w.x * pre, w.y * pre, w.z * pre, w.w * pre};
        uint32_t th[4], tl[4];
        uint32_t sum = 0u;   // mod 2^32: the constant offsets cancel below
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float q = e[j] * inv;
            const float t1 = __fadd_rn(q, kMagic);
            const float hq = __fsub_rn(t1, kMagic);
            const float r = __fmul_rn(__fsub_rn(q, hq), 254.0f);
            th[j] = __float_as_uint(t1);
            tl[j] = __float_as_uint(__fadd_rn(r, kMagic));
            sum += 254u * th[j] + tl[j];
        }
        hw[h2] = __byte_perm(__byte_perm(th[0], th[1], 0x0040), __byte_perm(th[2], th[3], 0x0040), 0x5410);
        lw[h2] = __byte_perm(__byte_perm(tl[0], tl[1], 0x0040), __byte_perm(tl[2], tl[3], 0x0040), 0x5410);
        sums[h2] = static_cast<int>(sum - 4u * 255u * kMagicBits);
    }
    if (!ok) hw[0] = hw[1] = lw[0] = lw[1] = 0u, sums[0] = sums[1] = 0;
    xq[lane] = make_uint4(hw[0], hw[1], lw[0], lw[1]);
    x4[lane] = make_int2(-32 * sums[0], -32 * sums[1]);
    const float u = ok ? (amax * pre) / 127.0f / 254.0f : (m == 0u ? 0.0f : amax);
    return make_float2(u, 1.0f / pre);
}

template <int BMAX, int RW, int ST>
__global__ void __launch_bounds__(kThreads) q6k_gemv_staged(const uint8_t *__restrict__ W, const float *__restrict__ x,
                                                           float *__restrict__ y, int N, int nb, int B, int tiles,
                                                           int sb)
{
    constexpr int TR = 8 * RW;                            // rows per tile: warp w takes rows w, w + 8, ...
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[ST];
    __shared__ int s_done[ST];
    __shared__ int s_abort;
    __shared__ int s_issued;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t RB = static_cast<size_t>(nb) * kBytes;   // row bytes
    const int pitch = q6_pitch(sb);
    const int stage_bytes = TR * pitch;
    const int nslices = (nb + sb - 1) / sb;
    // x area: per (batch row, block) 32 x 16 bytes of parts and 32 x 8 of sums, then the steps
    uint8_t *xa = smem + ST * stage_bytes;
    float2 *xup = reinterpret_cast<float2 *>(xa + static_cast<size_t>(B) * nb * kXItemBytes);
    const int my_tiles = (tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                         static_cast<int>(gridDim.x);
    const int total = my_tiles * nslices;
    const uint64_t policy = l2_policy_evict_first();
    // stage i of this CTA's schedule: tile blockIdx.x + (i / nslices) * gridDim.x, slice i % nslices
    auto issue = [&](int i) {
        const int slot = i % ST;
        const size_t tile = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(i / nslices) * gridDim.x;
        const int sl = i % nslices;
        const int j0 = sl * sb, j1 = min(nb, j0 + sb);
        uint32_t bytes = 0;
#pragma unroll
        for (int r = 0; r < TR; ++r) {
            const size_t start = (tile * TR + r) * RB + static_cast<size_t>(j0) * kBytes;
            const size_t end = start + static_cast<size_t>(j1 - j0) * kBytes;
            bytes += static_cast<uint32_t>(((end + 15) & ~static_cast<size_t>(15)) - (start & ~static_cast<size_t>(15)));
        }
        mbar_arrive_expect_tx(smem_u32(&full[slot]), bytes);
#pragma unroll
        for (int r = 0; r < TR; ++r) {
            const size_t start = (tile * TR + r) * RB + static_cast<size_t>(j0) * kBytes;
            const size_t end = start + static_cast<size_t>(j1 - j0) * kBytes;
            const size_t a0 = start & ~static_cast<size_t>(15);
            bulk_g2s(smem_u32(smem + slot * stage_bytes + r * pitch), W + a0,
                     static_cast<uint32_t>(((end + 15) & ~static_cast<size_t>(15)) - a0), smem_u32(&full[slot]), policy);
        }
    };
    if (tid == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            s_done[i] = 0;
        }
        s_abort = 0;
        fence_barrier_init();
        const int first = min(ST, total);
        for (int i = 0; i < first; ++i) issue(i);
        s_issued = first;
    }
    const int h = lane >> 4, c1 = (lane >> 3) & 1, l0 = 4 * (lane & 7);
    const int k_lo = 128 * h + 32 * c1 + l0;   // this lane's first low weight; +64 for the high ones
    // x -> int8 parts, one (batch row, block) per warp and round
    for (int it = warp; it < B * nb; it += kWarps) {
        const float *xb = x + static_cast<size_t>(it) * 256 + k_lo;   // row b = it / nb, block it % nb
        const float4 v0 = __ldg(reinterpret_cast<const float4 *>(xb));
        const float4 v1 = __ldg(reinterpret_cast<const float4 *>(xb + 64));
        uint8_t *item = xa + static_cast<size_t>(it) * kXItemBytes;
        const float2 up = q6_x_item(v0, v1, lane, reinterpret_cast<uint4 *>(item), reinterpret_cast<int2 *>(item + 512));
        if (lane == 0) xup[it] = up;
    }
    __syncthreads();
    const int ql_off = 4 * lane;
    const int qh_off = 128 + 32 * h + l0;
    const int sc_off = 192 + 8 * h + 2 * c1 + (l0 >> 4);   // scale of the low weights; +4 for the high ones
    const int qsh = 2 * c1;                                 // qh bits of the low weights; +4 for the high ones
    float acc[RW][BMAX];
    for (int i = 0; i < total; ++i) {
        const int ti = i / nslices, sl = i % nslices;
        const int tile = static_cast<int>(blockIdx.x) + ti * static_cast<int>(gridDim.x);
        if (sl == 0) {
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int b = 0; b < BMAX; ++b) acc[r][b] = 0.f;
        }
        const int slot = i % ST;
        const uint32_t phase = static_cast<uint32_t>((i / ST) & 1);
        if (!*(volatile int *)&s_abort && !mbar_wait_bounded(smem_u32(&full[slot]), phase, kWaitLimitNs)) {
            atomicOr(&g_q6k_error, 1u);
            s_abort = 1;
        }
        const int j0 = sl * sb, nj = min(nb, j0 + sb) - j0;
        const uint8_t *rowp[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const int tr = warp + 8 * r;
            const size_t start = (static_cast<size_t>(tile) * TR + tr) * RB + static_cast<size_t>(j0) * kBytes;
            rowp[r] = smem + slot * stage_bytes + tr * pitch + static_cast<int>(start & 15);
        }
#pragma unroll 2
        for (int j = 0; j < nj; ++j) {
            // this lane's x parts of block j0 + j, shared by the warp's RW rows
            uint4 xv[BMAX];
            int2 x4[BMAX];
            float xs[BMAX];
#pragma unroll
            for (int b = 0; b < BMAX; ++b) {
                // rows past B read row 0's parts (never used for an output)
                const int item = (b < B ? b : 0) * nb + j0 + j;
                const uint8_t *xi = xa + static_cast<size_t>(item) * kXItemBytes;
                xv[b] = reinterpret_cast<const uint4 *>(xi)[lane];
                x4[b] = reinterpret_cast<const int2 *>(xi + 512)[lane];
                const float2 up = xup[item];
                xs[b] = up.x * up.y;
            }
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const uint8_t *A = rowp[r] + j * kBytes;
                const uint32_t ql = lds_u16(A + ql_off) | (lds_u16(A + ql_off + 2) << 16);
                const uint32_t qh = lds_u16(A + qh_off) | (lds_u16(A + qh_off + 2) << 16);
                const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(lds_u16(A + 208))));
                const int sc_lo = static_cast<int8_t>(A[sc_off]);
                const int sc_hi = static_cast<int8_t>(A[sc_off + 4]);
                // q (0..63) of the four low and the four high weights, one per
                // byte: low nibble from ql, bits 4-5 from the lane's qh pair
                const uint32_t q_lo = and_or(ql, 0x0F0F0F0Fu, (qh << (4 - qsh)) & 0x30303030u);
                const uint32_t q_hi = and_or(ql >> 4, 0x0F0F0F0Fu, (qh >> qsh) & 0x30303030u);
#pragma unroll
                for (int b = 0; b < BMAX; ++b) {
                    const int t_lo = 254 * dp4a_us(q_lo, xv[b].x, 0) + dp4a_us(q_lo, xv[b].z, x4[b].x);
                    const int t_hi = 254 * dp4a_us(q_hi, xv[b].y, 0) + dp4a_us(q_hi, xv[b].w, x4[b].y);
                    const int ts = sc_lo * t_lo + sc_hi * t_hi;
                    acc[r][b] = fmaf(static_cast<float>(ts), d * xs[b], acc[r][b]);
                }
            }
        }
        // this warp is done with the slot: the last warp to finish refills it
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const int prev = atomicAdd(&s_done[slot], 1);
            if (prev % kWarps == kWarps - 1) {
                const int next = i + ST;
                if (next < total && !*(volatile int *)&s_abort) {
                    issue(next);
                    atomicAdd(&s_issued, 1);
                }
            }
        }
        if (sl == nslices - 1) {
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int b = 0; b < BMAX; ++b) {
                    if (b >= B) break;
                    float v = acc[r][b];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0 && !*(volatile int *)&s_abort)
                        y[static_cast<size_t>(b) * N + tile * TR + warp + 8 * r] = v;
                }
        }
    }
    // After a timed-out wait, wait (bounded) for the copies issued but not
    // consumed, so that none lands after the CTA has exited.
    __syncthreads();
    if (*(volatile int *)&s_abort && tid == 0) {
        for (int i = max(0, s_issued - ST); i < s_issued; ++i)
            if (!mbar_wait_bounded(smem_u32(&full[i % ST]), static_cast<uint32_t>((i / ST) & 1), kWaitLimitNs))
                break;
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
static cudaError_t q6k_launch(const uint8_t *W, const float *x, float *y, int N, int ldy, int nb, int B, int wpr,
                              int groups, int sms, size_t smem, cudaStream_t s)
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
    kern<<<grid, q6::kThreads, smem, s>>>(W, x, y, N, ldy, nb, B, wpr, groups);
    return cudaGetLastError();
}

template <int BMAX, int RW, int ST>
static cudaError_t q6k_launch_staged(const uint8_t *W, const float *x, float *y, int N, int nb, int B, int tiles,
                                     int sb, int sms, size_t smem, cudaStream_t s)
{
    auto kern = q6::q6k_gemv_staged<BMAX, RW, ST>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, q6::kThreads, smem);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(std::min<long long>(tiles, static_cast<long long>(sms) * std::max(occ, 1)));
    kern<<<grid, q6::kThreads, smem, s>>>(W, x, y, N, nb, B, tiles, sb);
    return cudaGetLastError();
}

// The direct kernel on rows [0, N) of W, output rows with stride ldy.
static cudaError_t q6k_direct(const uint8_t *W, const float *x, float *y, int N, int ldy, int nb, int batch, int sms,
                              cudaStream_t s)
{
    const int wpr = q6k_warps_per_row(N, nb, sms);
    const int rows_per_cta = q6::RPW * (q6::kWarps / wpr);
    const int groups = (N + rows_per_cta - 1) / rows_per_cta;
    // x staged in shared memory when it is small enough to leave room for six
    // or more CTAs per SM (a larger x there cost more in latency hiding than
    // it saved in loads: measured); persistent CTAs then load it once each
    const size_t xbytes = static_cast<size_t>(batch) * static_cast<size_t>(nb) * 256 * 4;
    const bool xs = xbytes <= 32 * 1024;
    if (batch == 1)
        return xs ? q6k_launch<1, true>(W, x, y, N, ldy, nb, batch, wpr, groups, sms, xbytes, s)
                  : q6k_launch<1, false>(W, x, y, N, ldy, nb, batch, wpr, groups, sms, 0, s);
    if (batch <= 4)
        return xs ? q6k_launch<4, true>(W, x, y, N, ldy, nb, batch, wpr, groups, sms, xbytes, s)
                  : q6k_launch<4, false>(W, x, y, N, ldy, nb, batch, wpr, groups, sms, 0, s);
    return xs ? q6k_launch<16, true>(W, x, y, N, ldy, nb, batch, wpr, groups, sms, xbytes, s)
              : q6k_launch<16, false>(W, x, y, N, ldy, nb, batch, wpr, groups, sms, 0, s);
}

unsigned int read_q6k_error()
{
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, q6::g_q6k_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    return v;
}

bool clear_q6k_error()
{
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(q6::g_q6k_error, &z, sizeof(z)) == cudaSuccess;
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
    const int n = static_cast<int>(N);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t *Wb = static_cast<const uint8_t *>(W);
    cudaError_t e = cudaSuccess;
    // Staged integer path (batch <= 4): whole tiles of 8 rows in K-slices of
    // up to 16 blocks, x converted into shared memory beside the ring (when
    // that takes at most 64 KB); the remaining N % 8 rows go to the direct
    // kernel.
    // Batch 1 takes two rows per warp when a row fits one 48 KB stage slice
    // (K up to 3584) and there is a whole 16-row tile; otherwise, like batch
    // 2-4, one row per warp in 28 KB stages (K up to 4096).
    auto slice = [&](int rw, int skb) {
        return std::max(1, std::min(nb, ((skb * 1024) / (8 * rw) - 30) / q6::kBytes));
    };
    const bool pair = batch == 1 && slice(q6::kRW1, q6::kStageKB1) == nb && n >= 8 * q6::kRW1;
    const int RW = pair ? q6::kRW1 : q6::kRW4;
    const int ST = pair ? q6::kStages1 : q6::kStages4;
    const int tiles = n / (8 * RW);
    const size_t xbytes = static_cast<size_t>(batch) * nb * (q6::kXItemBytes + 8);
    // (rows longer than one slice, e.g. K = 18944, measured faster on the
    // direct kernel: 27 against 31 us)
    const int sb = slice(RW, pair ? q6::kStageKB1 : q6::kStageKB4);
    if (batch <= 4 && tiles > 0 && xbytes <= 64 * 1024 && sb == nb) {
        const size_t smem = static_cast<size_t>(ST) * 8 * RW * q6::q6_pitch(sb) + xbytes;
        if (pair)
            e = q6k_launch_staged<1, q6::kRW1, q6::kStages1>(Wb, x, y, n, nb, batch, tiles, sb, sms, smem, s);
        else if (batch == 1)
            e = q6k_launch_staged<1, q6::kRW4, q6::kStages4>(Wb, x, y, n, nb, batch, tiles, sb, sms, smem, s);
        else
            e = q6k_launch_staged<4, q6::kRW4, q6::kStages4>(Wb, x, y, n, nb, batch, tiles, sb, sms, smem, s);
        const int done = tiles * 8 * RW;
        if (e == cudaSuccess && done < n)
            e = q6k_direct(Wb + static_cast<size_t>(done) * nb * q6::kBytes, x, y + done, n - done, n, nb, batch, sms, s);
    } else {
        e = q6k_direct(Wb, x, y, n, n, nb, batch, sms, s);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4K_ERR_CUDA;
    }
    return Q4K_OK;
}

}  // namespace q4k
